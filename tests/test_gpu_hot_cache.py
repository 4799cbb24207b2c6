"""Parity of the cross-step hot cache (qsa_hot_cache_fetch, through the C ABI)
with the fp64 oracle's hot_cache_step.

Bars: after every step the slot table of every unit equals the oracle's, bit
for bit (which tokens hold which hot rows, which went cold); every hot row
the oracle filled holds the host row of its token, byte for byte; and decode
steps that fetch into the hot cache produce the oracle's selections and
attention (attention within 2e-3) while the oracle reads cold rows from host
memory.  The oracle is fed only generator bytes and the test's own
selections, never what the kernels wrote.
"""
import numpy as np
import pytest
import torch

import sparse_attention_decode_qsa_gb300 as Q
from oracle import qsa_oracle as O
from sparse_attention_decode_qsa_gb300 import synth, workloads
from tests import qsa_check as QC

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    Q.lib()


def _clean(wl):
    st, det = wl.cache.poll_error()
    assert st == 0, f"device error word {st} detail {det}"


class _OracleUnit:
    """The oracle's view of one unit's slot row and hot-cache state."""

    def __init__(self, wl, l, r):
        info = wl.cache.request_info(wl.handles[r])
        self.n = wl.ctxs[r]
        self.slot = QC.oracle_slot_row(wl, l, r)
        self.hot = info.hot_row_base >= 0
        H = wl.cache.hot_rows
        self.hot_base = info.hot_row_base + l * H if self.hot else -1
        self.owner = np.full(H, -1, dtype=np.int32)
        self.cursor = 0

    def step(self, sel_blocks):
        if not self.hot:
            return []
        toks = O.selected_tokens(sel_blocks, self.n)
        self.slot, self.owner, self.cursor, fills = O.hot_cache_step(
            toks, self.slot, self.owner, self.cursor, self.hot_base)
        return fills


def _random_selection(rng, n, k_max, prev, keep):
    nb = (n + 3) // 4
    k = int(rng.integers(0, min(k_max, nb) + 1))
    kept = [b for b in prev if rng.random() < keep][:k]
    rest = np.setdiff1d(np.arange(nb), kept)
    extra = rng.choice(rest, k - len(kept), replace=False) if k > len(kept) else []
    sel = np.sort(np.concatenate([np.asarray(kept, dtype=np.int64), np.asarray(extra, dtype=np.int64)]))
    if rng.random() < 0.3 and nb - 1 not in sel and len(sel) < min(k_max, nb):
        sel = np.sort(np.append(sel, nb - 1))           # the ragged last block
    return sel.astype(np.int32)


@pytest.mark.parametrize("kv_format", [Q.KV_BF16, Q.KV_FP8])
def test_hot_cache_fetch_matches_the_oracle_over_drifting_steps(kv_format):
    budget, H, ring = 512, 600, 256
    ctxs = [6001, 9000, 3000, 1500]
    placements = [Q.KV_HOST_RING, Q.KV_HOST, Q.KV_HOST_RING, Q.KV_HBM]
    L = 2
    wl = workloads.build(L, ctxs, placements, lambda l, r, n: [], budget=budget, ring=ring,
                         staging_rows=8, seed=31, hot_rows=H, kv_format=kv_format)
    try:
        c, R = wl.cache, len(ctxs)
        rng = np.random.default_rng(31)
        units = {(l, r): _OracleUnit(wl, l, r) for l in range(L) for r in range(R)}
        prev = {key: [] for key in units}
        k_max = budget // 4
        host_np = [h.numpy() if h is not None else None for h in wl.host]
        for step in range(14):
            keep = [1.0, 0.9, 0.5, 0.0][step % 4]
            sel = torch.zeros(L * R, k_max, dtype=torch.int32)
            nsel = torch.zeros(L * R, dtype=torch.int32)
            for (l, r), ou in units.items():
                s = _random_selection(rng, ctxs[r], k_max, prev[(l, r)], keep)
                prev[(l, r)] = list(s)
                sel[wl.unit(l, r), :len(s)] = torch.from_numpy(s)
                nsel[wl.unit(l, r)] = len(s)
            wl.sel.copy_(sel.cuda())
            wl.nsel.copy_(nsel.cuda())
            for l in range(L):
                sl = slice(l * R, (l + 1) * R)
                c.hot_cache_fetch(wl.handles, l, 1, wl.sel[sl], wl.nsel[sl], budget)
            torch.cuda.synchronize()
            _clean(wl)
            for (l, r), ou in units.items():
                u = wl.unit(l, r)
                fills = ou.step(sel[u, :int(nsel[u])].numpy())
                h = wl.handles[r]
                got = c.slot_table[h.index, l, :ctxs[r]].cpu().numpy()
                assert np.array_equal(got, ou.slot), (step, l, r)
                if fills:
                    rows = torch.tensor([row for _, row in fills], dtype=torch.int64, device="cuda")
                    got_rows = c.pool[rows].cpu().numpy()
                    want = np.stack([host_np[r][l, t] for t, _ in fills])
                    assert np.array_equal(got_rows, want), (step, l, r)
    finally:
        wl.close()


@pytest.mark.parametrize("fold", [False, True])
@pytest.mark.parametrize("kv_format", [Q.KV_BF16, Q.KV_FP8])
def test_hot_cache_decode_steps_match_the_oracle(kv_format, fold):
    """Decode steps (score, top-k, fetch, attention) over a host-ring cache
    with hot rows (BF16 and FP8 rows), the selection drifting between steps:
    selections and attention match the oracle, which reads every cold row
    from host memory, and the slot tables follow the oracle's hot-cache
    state.  With fold, the step plans the hot rows (qsa_hot_cache_plan) and
    the attention copies the misses into them."""
    L, R, n, ring, H, seed = 2, 2, 40000, 2048, 2048, 41
    wl = workloads.build(L, [n] * R, [Q.KV_HOST_RING] * R,
                         lambda l, r, n: synth.planted_hot_cold(n // 4, 512, ring // 4,
                                                                synth.mix_seed(seed, 90, l, r)),
                         ring=ring, staging_rows=8, seed=seed, hot_rows=H, kv_format=kv_format)
    wl.fold_fill = fold
    try:
        units = {(l, r): _OracleUnit(wl, l, r) for l in range(L) for r in range(R)}
        for step, frac in enumerate([0.0, 0.0, 0.25, 1.0, 0.1]):
            if frac:
                wl.drift(frac, synth.mix_seed(seed, 500, step))
            wl.step()
            torch.cuda.synchronize()
            _clean(wl)
            for (l, r), ou in units.items():
                res = QC.check_unit(wl, l, r)
                ou.step(res["ref"]["sel"])
                h = wl.handles[r]
                got = wl.cache.slot_table[h.index, l, :n].cpu().numpy()
                assert np.array_equal(got, ou.slot), (step, l, r)
                toks = res["ref"]["tokens"]
                assert np.all(got[toks] >= 0)              # every selected row now in HBM
    finally:
        wl.close()


def _same(wl, out_lse, slots, step):
    # the micro-batched step splits attention differently: equal up to the
    # order of the split-K merge
    assert torch.allclose(wl.out, out_lse[0], rtol=1e-5, atol=1e-6), step
    assert torch.allclose(wl.lse, out_lse[1], rtol=1e-6, atol=1e-6), step
    assert torch.equal(wl.cache.slot_table, slots), step


@pytest.mark.parametrize("fold", [False, True])
def test_hot_cache_pipelined_graph_step_matches_sequential_steps(fold):
    """The captured two-micro-batch step with fetches (or, with fold, plans
    whose copies ride on the attention) gives the same outputs and slot
    tables as eager sequential steps with fetches on an identical workload,
    over steps whose selection drifts."""
    L, R, n, ring, H, seed = 2, 4, 30000, 1024, 2048, 43

    def make():
        return workloads.build(L, [n] * R, [Q.KV_HOST_RING] * R,
                               lambda l, r, n: synth.planted_hot_cold(n // 4, 512, ring // 4,
                                                                      synth.mix_seed(seed, 90, l, r)),
                               ring=ring, staging_rows=8, seed=seed, hot_rows=H)
    a = make()
    try:
        outs, slots = [], []
        for step in range(4):
            if step:
                a.drift(0.5, synth.mix_seed(seed, 600, step))
            a.step()
            torch.cuda.synchronize()
            _clean(a)
            outs.append((a.out.clone(), a.lse.clone()))
            slots.append(a.cache.slot_table.clone())
    finally:
        a.close()
    b = make()
    b.fold_fill = fold
    try:
        streams = b.make_streams(2)
        b.step_pipelined(streams)                 # step 0 (eager, sets kernel attributes)
        torch.cuda.synchronize()
        _clean(b)
        _same(b, outs[0], slots[0], 0)
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        b.drift(0.5, synth.mix_seed(seed, 600, 1))
        with torch.cuda.graph(g, stream=cap):
            b.step_pipelined(streams)             # capture only: nothing runs
        torch.cuda.synchronize()
        for step in range(1, 4):
            if step > 1:
                b.drift(0.5, synth.mix_seed(seed, 600, step))
            g.replay()
            torch.cuda.synchronize()
            _clean(b)
            _same(b, outs[step], slots[step], step)
    finally:
        b.close()


def test_hot_cache_rejects_bad_selections():
    wl = workloads.build(1, [5000], [Q.KV_HOST_RING], lambda l, r, n: [], budget=512, ring=256,
                         staging_rows=8, seed=44, hot_rows=512)
    try:
        c = wl.cache
        before = c.slot_table.clone()
        wl.sel[0, :2] = torch.tensor([3, 5000], dtype=torch.int32)     # block 5000 is past the end
        wl.nsel[0] = 2
        c.hot_cache_fetch(wl.handles, 0, 1, wl.sel, wl.nsel, 512)
        torch.cuda.synchronize()
        st, _ = c.poll_error()
        assert st == Q.ERR_BAD_BLOCK
        assert torch.equal(c.slot_table, before)
        wl.nsel[0] = 10000                                             # more than budget/4
        c.hot_cache_fetch(wl.handles, 0, 1, wl.sel, wl.nsel, 512)
        torch.cuda.synchronize()
        st, _ = c.poll_error()
        assert st == Q.ERR_BAD_BLOCK
        assert torch.equal(c.slot_table, before)
        with pytest.raises(Q.QsaError) as e:
            c.hot_cache_fetch(wl.handles, 0, 1, wl.sel, wl.nsel, 1024)   # above the config budget
        assert e.value.status == Q.ERR_INVALID_ARG
    finally:
        wl.close()


def test_hot_cache_state_starts_fresh_for_a_reissued_request():
    """A request that ends hands its hot rows back; the request admitted in
    its slot starts with every hot row free and the cursor at row 0 (the
    oracle's fresh state), even when it gets the same pool rows."""
    budget, H, ring = 512, 512, 256
    wl = workloads.build(1, [7000, 5000], [Q.KV_HOST_RING] * 2, lambda l, r, n: [], budget=budget,
                         ring=ring, staging_rows=8, seed=45, hot_rows=H)
    try:
        c = wl.cache
        rng = np.random.default_rng(45)
        k_max = budget // 4

        def fetch_random(units):
            sel = torch.zeros(2, k_max, dtype=torch.int32)
            nsel = torch.zeros(2, dtype=torch.int32)
            for r in range(2):
                s = _random_selection(rng, wl.ctxs[r], k_max, [], 0.0)
                sel[r, :len(s)] = torch.from_numpy(s)
                nsel[r] = len(s)
            wl.sel.copy_(sel.cuda())
            wl.nsel.copy_(nsel.cuda())
            c.hot_cache_fetch(wl.handles, 0, 1, wl.sel, wl.nsel, budget)
            torch.cuda.synchronize()
            _clean(wl)
            for r in range(2):
                units[r].step(sel[r, :int(nsel[r])].numpy())

        units = [_OracleUnit(wl, 0, r) for r in range(2)]
        for _ in range(3):
            fetch_random(units)
        old_hot = c.request_info(wl.handles[0]).hot_row_base
        wl.reissue(0, 6000, Q.KV_HOST_RING, seed=46)
        assert c.request_info(wl.handles[0]).hot_row_base == old_hot      # same rows reused
        units[0] = _OracleUnit(wl, 0, 0)
        for _ in range(3):
            fetch_random(units)
            for r in range(2):
                got = c.slot_table[wl.handles[r].index, 0, :wl.ctxs[r]].cpu().numpy()
                assert np.array_equal(got, units[r].slot), r
    finally:
        wl.close()


@pytest.mark.parametrize("kv_format", [Q.KV_BF16, Q.KV_FP8])
def test_hot_cache_plan_then_attention_matches_the_oracle(kv_format):
    """qsa_hot_cache_plan followed by qsa_sparse_decode_attn, over drifting
    random selections: after each attention the slot tables equal the
    oracle's hot_cache_step state and every row the oracle fills holds its
    host row, byte for byte (the attention wrote it); the attention equals
    the oracle's attention over the selected tokens' host rows; a second
    attention without a new plan reads the filled rows from HBM and gives
    the same result bit for bit."""
    budget, H, ring = 512, 600, 256
    ctxs = [6001, 9000, 3000]
    placements = [Q.KV_HOST_RING, Q.KV_HOST, Q.KV_HOST_RING]
    L = 2
    wl = workloads.build(L, ctxs, placements, lambda l, r, n: [], budget=budget, ring=ring,
                         staging_rows=8, seed=47, hot_rows=H, kv_format=kv_format)
    try:
        c, R = wl.cache, len(ctxs)
        fp8 = kv_format == Q.KV_FP8
        rng = np.random.default_rng(47)
        units = {(l, r): _OracleUnit(wl, l, r) for l in range(L) for r in range(R)}
        prev = {key: [] for key in units}
        k_max = budget // 4
        host_np = [h.numpy() for h in wl.host]
        for step in range(8):
            keep = [1.0, 0.9, 0.5, 0.0][step % 4]
            sel = torch.zeros(L * R, k_max, dtype=torch.int32)
            nsel = torch.zeros(L * R, dtype=torch.int32)
            for (l, r), ou in units.items():
                s_ = _random_selection(rng, ctxs[r], k_max, prev[(l, r)], keep)
                prev[(l, r)] = list(s_)
                sel[wl.unit(l, r), :len(s_)] = torch.from_numpy(s_)
                nsel[wl.unit(l, r)] = len(s_)
            wl.sel.copy_(sel.cuda())
            wl.nsel.copy_(nsel.cuda())
            for l in range(L):
                sl = slice(l * R, (l + 1) * R)
                c.hot_cache_plan(wl.handles, l, 1, wl.sel[sl], wl.nsel[sl], budget)
                c.sparse_decode_attn(wl.handles, l, 1, wl.q[sl], wl.sel[sl], wl.nsel[sl], budget,
                                     None, wl.softmax_scale, wl.out[sl], wl.lse[sl])
            torch.cuda.synchronize()
            _clean(wl)
            out1, lse1 = wl.out.clone(), wl.lse.clone()
            for l in range(L):
                sl = slice(l * R, (l + 1) * R)
                c.sparse_decode_attn(wl.handles, l, 1, wl.q[sl], wl.sel[sl], wl.nsel[sl], budget,
                                     None, wl.softmax_scale, wl.out[sl], wl.lse[sl])
            torch.cuda.synchronize()
            _clean(wl)
            assert torch.equal(out1, wl.out) and torch.equal(lse1, wl.lse), step
            for (l, r), ou in units.items():
                u = wl.unit(l, r)
                blocks = sel[u, :int(nsel[u])].numpy()
                fills = ou.step(blocks)
                h = wl.handles[r]
                got = c.slot_table[h.index, l, :ctxs[r]].cpu().numpy()
                assert np.array_equal(got, ou.slot), (step, l, r)
                if fills:
                    rows = torch.tensor([row for _, row in fills], dtype=torch.int64, device="cuda")
                    got_rows = c.pool[rows].cpu().numpy()
                    want = np.stack([host_np[r][l, t] for t, _ in fills])
                    assert np.array_equal(got_rows, want), (step, l, r)
                toks = O.selected_tokens(blocks, ctxs[r])
                o_ref, lse_ref = O.decode_attention(QC.bits16(wl.q[u]), host_np[r][l][toks],
                                                    wl.softmax_scale, "fp8" if fp8 else "bf16")
                assert np.abs(out1[u].cpu().double().numpy() - o_ref).max() <= QC.ATTN_TOL, (step, l, r)
                assert np.abs(lse1[u].cpu().double().numpy() - lse_ref).max() <= QC.ATTN_TOL, (step, l, r)
    finally:
        wl.close()
