"""CPU tests of the seeded input generators' selection-drift helpers (the
inputs of the benchmark's drift measurement): the drift moves exactly the
asked share of the planted blocks inside the range to unplanted blocks of
the same range, keeps the rest, and undoing a plant restores the scales bit
for bit."""
import numpy as np
import torch

from sparse_attention_decode_qsa_gb300 import synth


def test_drift_blocks_moves_the_asked_share_inside_the_range():
    planted = synth.planted_hot_cold(65536, 512, 1024, seed=3)
    lo, hi = 0, 65536 - 1024
    inside = planted[(planted >= lo) & (planted < hi)]
    for frac in (0.0, 0.1, 0.25, 1.0):
        dropped, added, now = synth.drift_blocks(planted, lo, hi, frac, seed=7)
        k = int(round(frac * inside.numel()))
        assert dropped.numel() == k and added.numel() == k
        assert now.numel() == planted.numel() and torch.equal(now, now.unique())
        assert bool(torch.isin(dropped, inside).all())
        assert not bool(torch.isin(added, planted).any())
        assert bool(((added >= lo) & (added < hi)).all())
        outside = planted[(planted < lo) | (planted >= hi)]
        assert bool(torch.isin(outside, now).all())            # blocks outside the range stay
        keep = planted[~torch.isin(planted, dropped)]
        assert torch.equal(torch.sort(torch.cat([keep, added])).values, now)
    d1, a1, _ = synth.drift_blocks(planted, lo, hi, 0.5, seed=9)
    d2, a2, _ = synth.drift_blocks(planted, lo, hi, 0.5, seed=9)
    assert torch.equal(d1, d2) and torch.equal(a1, a2)           # seeded


def test_drift_blocks_when_the_range_is_nearly_full():
    planted = torch.arange(0, 10)
    dropped, added, now = synth.drift_blocks(planted, 0, 12, 1.0, seed=1)
    assert dropped.numel() == 2 and added.numel() == 2           # only two free blocks
    assert set(added.tolist()) == {10, 11}
    assert now.numel() == 10


def test_unplant_restores_plant_exactly():
    g = torch.Generator().manual_seed(5)
    n = 4099                                                     # ragged last block
    sc = (torch.rand(n, generator=g) * torch.exp2(torch.randint(-20, 4, (n,), generator=g).float())).half()
    sc[:8] = torch.tensor([0.0, -0.0, 6.0e-8, 1.0e-5, 0.5, 1.0, 800.0, 1000.0]).half()
    before = sc.clone()
    blocks = [0, 1, 5, 17, 1024]                                 # 1024: the partial last block
    synth.plant(sc, blocks, n)
    assert not torch.equal(sc.view(torch.int16), before.view(torch.int16))
    synth.unplant(sc, blocks, n)
    assert np.array_equal(sc.view(torch.int16).numpy(), before.view(torch.int16).numpy())


def test_planting_recipes_match_their_definitions():
    """The planting recipes of the workloads: uniform distinct blocks; half
    of the planted blocks inside the tail ring and half before it (the 256K
    config); sinks 0-3 plus a 50/50 mix of a recency Zipf(1.1) law and a
    uniform law (the 1M config)."""
    u = synth.planted_uniform(1000, 300, seed=2)
    assert u.numel() == 300 and u.unique().numel() == 300 and int(u.min()) >= 0 and int(u.max()) < 1000
    assert synth.planted_uniform(10, 300, seed=2).numel() == 10

    n_blocks, tail = 65536, 1024
    hc = synth.planted_hot_cold(n_blocks, 512, tail, seed=3)
    assert hc.numel() == 512 and hc.unique().numel() == 512
    assert int((hc >= n_blocks - tail).sum()) == 256 and int((hc < n_blocks - tail).sum()) == 256
    small = synth.planted_hot_cold(600, 512, 1024, seed=3)           # tail covers every block
    assert small.numel() == 512 and int(small.max()) < 600

    nb = 262144
    z = synth.planted_zipf_sinks(nb, 512, seed=4)
    assert z.numel() == 512 and z.unique().numel() == 512 and int(z.max()) < nb
    assert set(range(4)) <= set(z.tolist())
    newest_percent = int((z >= nb - nb // 100).sum())
    assert 100 <= newest_percent <= 400            # the recency law puts ~200 of 508 there
    assert int((z < nb // 2).sum()) >= 100          # the uniform half spreads over the context


def test_ragged_contexts_are_log_uniform_multiples():
    ctx = synth.log_uniform_contexts(64, 4096, 262144, seed=5)
    ctx = [int(c) for c in ctx]
    assert all(c % 4 == 0 and 4096 <= c <= 262144 for c in ctx)
    assert min(ctx) < 16384 and max(ctx) > 65536   # spread over the decades, not clustered
    assert ctx == [int(c) for c in synth.log_uniform_contexts(64, 4096, 262144, seed=5)]


def test_skewed_index_query_spans_the_stated_range():
    q, w = synth.index_query_skewed(seed=5)
    a = q.abs().double()
    assert q.shape == (8, 64) and w.shape == (8,)
    assert float(a.max()) <= 1.0 and float(a.min()) >= 2.0 ** -12
    assert float(a.max()) > 0.5 and float(a.min()) < 2.0 ** -11      # both ends reached
    assert 0.3 < float((q > 0).double().mean()) < 0.7                 # random signs
    q2, _ = synth.index_query_skewed(seed=5)
    assert torch.equal(q, q2)
