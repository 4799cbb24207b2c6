"""Parity of the CUDA library (through its C ABI) with the fp64 oracle.

Bars: selected block ids bit-exact on inputs whose fp64 boundary gap is at
least 1e-3 (asserted per unit); gathered rows byte-exact; attention out and
lse within 2e-3 max abs; block scores within 1e-5 of sum_h w_h sc
sum_d |q k| (the fp32 accumulation bound, with margin).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import sparse_attention_decode_qsa_gb300 as Q
from oracle import qsa_oracle as O
from sparse_attention_decode_qsa_gb300 import synth, workloads
from tests import qsa_check as QC

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    Q.lib()


def _clean(wl):
    st, det = wl.cache.poll_error()
    assert st == 0, f"device error word {st} detail {det}"


def test_tiny_end_to_end():
    wl = workloads.tiny()
    try:
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        res = QC.check_unit(wl, 0, 0)
        assert res["ref"]["sel"].tolist() == wl.planted[0][0].tolist()
    finally:
        wl.close()


def test_c128k_twelve_layers():
    """12 layers x 131072 tokens, KV in HBM; every layer checked."""
    wl = workloads.c128k()
    try:
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        sels = []
        for l in range(12):
            QC.check_unit(wl, l, 0)
            sels.append(tuple(wl.sel[l].cpu().tolist()))
        assert len(set(sels)) == 12       # the layers select on their own
    finally:
        wl.close()


def _run_select(blk_rows, ctxs, budget):
    """Select on given fp32 block scores, one unit per row."""
    cap = max(ctxs)
    c = Q.Cache(n_layers=1, max_requests=len(ctxs), ctx_capacity=cap,
                hbm_pool_rows=sum(ctxs) + 8, budget_tokens=max(budget, 4), staging_rows=0,
                device="cuda")
    try:
        hs = [c.request_begin(n, Q.KV_HBM) for n in ctxs]
        stride = (cap + 3) // 4
        blk = torch.full((len(ctxs), stride), float("nan"), dtype=torch.float32)
        for i, row in enumerate(blk_rows):
            blk[i, :len(row)] = torch.as_tensor(row, dtype=torch.float32)
        blk = blk.cuda()
        sel = torch.full((len(ctxs), budget // 4), -7, dtype=torch.int32, device="cuda")
        nsel = torch.empty(len(ctxs), dtype=torch.int32, device="cuda")
        c.select_c4_topk(hs, 0, 1, blk, budget, sel, nsel)
        torch.cuda.synchronize()
        return sel.cpu().numpy(), nsel.cpu().numpy()
    finally:
        c.close()


def test_topk_hand_worked_cases():
    cases = json.load(open(os.path.join(GOLDEN, "c4_topk_hand.json")))["cases"]
    for case in cases:
        n = len(case["token_scores"])
        sel, nsel = _run_select([case["blocks"]], [n], case["budget"])
        k = int(nsel[0])
        assert sel[0, :k].tolist() == case["selected"], case["name"]


def test_topk_bit_exact_on_any_fp32_scores():
    """The selection rule applied to the GPU's own fp32 inputs: identical to
    the oracle's selection of the same values, ties and signed zeros
    included, for contexts from 1 token to 1M tokens."""
    rng = np.random.default_rng(17)
    ctxs, rows, budgets = [], [], []
    for kind in range(10):
        n = int([1, 7, 4096, 8191, 65536, 131072, 262144, 1048576, 30000, 2049][kind])
        nb = (n + 3) // 4
        if kind % 3 == 0:
            v = rng.integers(-3, 4, size=nb).astype(np.float32)        # heavy ties
            v[rng.random(nb) < 0.1] = -0.0
        elif kind % 3 == 1:
            v = rng.standard_normal(nb).astype(np.float32) * 30
        else:
            v = np.round(rng.standard_normal(nb) * 4).astype(np.float32) / 8   # coarse ties
        ctxs.append(n)
        rows.append(v)
    # a call's largest unit sets the keys each cluster CTA holds: once with
    # the 1M-token unit (32768 keys per CTA), once without it (8192); heavy
    # ties also push some units onto the general path (boundary bin larger
    # than the candidate buffer)
    small = [i for i, n in enumerate(ctxs) if n <= 262144]
    for budget in (4, 2048, 8192):
        for pick in (list(range(len(ctxs))), small):
            sel, nsel = _run_select([rows[i] for i in pick], [ctxs[i] for i in pick], budget)
            for j, i in enumerate(pick):
                ref = O.select_blocks(rows[i].astype(np.float64), budget)
                assert int(nsel[j]) == len(ref)
                assert np.array_equal(sel[j, :len(ref)], ref), (ctxs[i], budget, len(pick))


def test_topk_small_boundary_bin_with_ties():
    """At most 32 keys in the bin of the first 11-bit digit that holds the
    K-th largest score, the case the planted workloads meet (there the K-th
    score is alone in its bin), which the top-k settles by ranking the few
    candidates directly: ties at the threshold, distinct values above it in
    the same bin, and bins of 32 and 33 keys (both sides of that switch).
    131072 tokens (8 CTAs of 4096 blocks), K = 512, bin keys spread over
    the CTAs; compared with the oracle's selection."""
    rng = np.random.default_rng(29)
    n, budget = 131072, 2048
    nb, K = n // 4, budget // 4

    def digit(x):   # first 11 bits of the order-preserving key of a positive float
        return int((np.float32(x).view(np.uint32) | np.uint32(0x80000000)) >> np.uint32(21))

    assert len({digit(x) for x in (2.0, 2.125, 2.25, 2.375)}) == 1
    assert digit(2.5) != digit(2.0) and digit(0.001) != digit(2.0)
    for n_top, n_eq, n_other in [(500, 20, 8), (511, 1, 0), (492, 24, 8), (492, 25, 8), (480, 32, 0),
                                 (510, 3, 29), (505, 10, 10)]:
        v = np.full(nb, 0.001, np.float32)
        top = rng.choice(nb, n_top, replace=False)
        v[top] = 1000 + np.arange(n_top, dtype=np.float32)
        rest = np.setdiff1d(np.arange(nb), top)
        pos = rng.choice(rest, n_eq + n_other, replace=False)
        v[pos[:n_eq]] = 2.0
        v[pos[n_eq:]] = rng.choice(np.array([2.125, 2.25, 2.375], np.float32), n_other)
        # the K-th largest lies in the bin of 2.0, which holds n_eq + n_other keys
        assert n_top < K <= n_top + n_eq + n_other
        sel, nsel = _run_select([v], [n], budget)
        ref = O.select_blocks(v.astype(np.float64), budget)
        assert int(nsel[0]) == len(ref) == K
        assert np.array_equal(sel[0, :K], ref), (n_top, n_eq, n_other)


def test_topk_units_on_different_paths_in_one_launch():
    """One launch whose clusters take different paths: a boundary bin of one
    key and one of 28 keys with ties (ranked directly), one of 40 keys (the
    radix passes over the candidates), heavy ties (the general path), and a
    1M-token unit with a one-key bin (a slice of 32768 keys, so warp ranges
    of 2048 in the candidate walk).  Each unit against the oracle."""
    rng = np.random.default_rng(31)
    budget = 2048
    K = budget // 4

    def planted(nb, n_top, n_eq, n_other):
        v = np.full(nb, 0.001, np.float32)
        top = rng.choice(nb, n_top, replace=False)
        v[top] = 1000 + np.arange(n_top, dtype=np.float32)
        rest = np.setdiff1d(np.arange(nb), top)
        pos = rng.choice(rest, n_eq + n_other, replace=False)
        v[pos[:n_eq]] = 2.0
        v[pos[n_eq:]] = rng.choice(np.array([2.125, 2.25, 2.375], np.float32), n_other)
        return v

    ctxs = [131072, 262144, 131072, 65536, 1048576]
    rows = [planted(ctxs[0] // 4, 511, 1, 0),
            planted(ctxs[1] // 4, 500, 20, 8),
            planted(ctxs[2] // 4, 490, 30, 10),
            rng.integers(-3, 4, size=ctxs[3] // 4).astype(np.float32),
            planted(ctxs[4] // 4, 511, 1, 0)]
    sel, nsel = _run_select(rows, ctxs, budget)
    for j, v in enumerate(rows):
        ref = O.select_blocks(v.astype(np.float64), budget)
        assert int(nsel[j]) == len(ref) == K
        assert np.array_equal(sel[j, :K], ref), ctxs[j]


def test_topk_boundary_bin_crowded_into_one_cta():
    """The boundary bin of the first 11-bit digit holds few keys overall (600,
    within the 2048 the CTAs finish the select on) but all in one CTA's slice,
    more than that CTA's 256 candidate slots: the call must take the general
    path.  Also the same keys spread over every slice (the usual path), and
    crowded into the last CTA.  Each equals the oracle's selection."""
    rng = np.random.default_rng(5)
    nb = 8192                       # 8 CTA slices of 1024 blocks
    S = nb // 8
    rows = []
    for where in ("first", "spread", "last"):
        v = np.full(nb, 0.001, np.float32)
        lo, hi = {"first": (0, S), "spread": (0, nb), "last": (nb - S, nb)}[where]
        inbin = rng.choice(np.arange(lo, hi), 600, replace=False)
        rest = np.setdiff1d(np.arange(nb), inbin)
        above = rng.choice(rest[rest >= S] if where != "last" else rest[rest < nb - S], 300,
                           replace=False)
        v[above] = 100.0 + rng.random(300).astype(np.float32)   # far above the bin
        # 600 distinct keys sharing their top 11 bits (1.0 .. 1.0006)
        v[inbin] = np.float32(1.0) + rng.permutation(600).astype(np.float32) * np.float32(2 ** -20)
        rows.append(v)
    sel, nsel = _run_select(rows, [4 * nb] * 3, 2048)
    for j, v in enumerate(rows):
        ref = O.select_blocks(v.astype(np.float64), 2048)
        assert int(nsel[j]) == len(ref) == 512
        assert np.array_equal(sel[j, :len(ref)], ref), j


def _host_ring_workload(n_req=2, n_layers=2, n=20000, seed=5):
    return workloads.build(n_layers, [n] * n_req, [Q.KV_HOST_RING] * n_req,
                           lambda l, r, n: synth.planted_hot_cold(n // 4, 512, 1024,
                                                                  synth.mix_seed(seed, 90, l, r)),
                           seed=seed)


def test_host_ring_gather_and_attention_modes():
    """Host history + HBM tail ring: selection and attention match the
    oracle; gathered rows are byte-exact; attention read through the slot
    table equals attention over the gathered rows to fp32 rounding (the two
    modes may spread the splits over a different number of CTAs, which
    changes only the merge order)."""
    wl = _host_ring_workload()
    try:
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        refs = {}
        for l in range(2):
            for r in range(2):
                refs[(l, r)] = QC.check_unit(wl, l, r)["ref"]
        out_direct = wl.out.clone()
        lse_direct = wl.lse.clone()
        budget = wl.budget
        for l in range(2):
            sl = slice(l * 2, (l + 1) * 2)
            g = torch.empty(2, budget, 2048, dtype=torch.uint8, device="cuda")
            nrows = torch.empty(2, dtype=torch.int32, device="cuda")
            wl.cache.gather_rows(wl.handles, l, 1, wl.sel[sl], wl.nsel[sl], budget, g, nrows)
            wl.cache.sparse_decode_attn(wl.handles, l, 1, wl.q[sl], wl.sel[sl], wl.nsel[sl], budget,
                                        g, wl.softmax_scale, wl.out[sl], wl.lse[sl])
            torch.cuda.synchronize()
            for r in range(2):
                ref = refs[(l, r)]
                m = len(ref["tokens"])
                assert int(nrows[r]) == m
                assert np.array_equal(g[r, :m].cpu().numpy(), ref["rows"])
        _clean(wl)
        assert torch.allclose(out_direct, wl.out, rtol=1e-5, atol=1e-6)
        assert torch.allclose(lse_direct, wl.lse, rtol=1e-6, atol=1e-6)
    finally:
        wl.close()


def test_dense_path_and_ragged_contexts():
    """Contexts at or below the budget take every block (dense attention);
    ragged contexts mask the missing tokens of the last block."""
    ctxs = [1, 3, 4, 10, 1000, 2047, 2048, 2049, 6001]
    wl = workloads.build(1, ctxs, [Q.KV_HBM] * len(ctxs),
                         lambda l, r, n: synth.planted_uniform((n + 3) // 4, min(512, (n + 3) // 4),
                                                               synth.mix_seed(6, r)),
                         staging_rows=0, seed=6)
    try:
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        for r, n in enumerate(ctxs):
            res = QC.check_unit(wl, 0, r)
            if n <= 2048:
                assert res["ref"]["tokens"].tolist() == list(range(n))
    finally:
        wl.close()


def test_slot_remap_to_staging_is_invisible():
    """Moving selected cold rows into staging rows (bytes copied, slot table
    updated) changes neither the selection nor the attention output."""
    wl = _host_ring_workload(n_req=1, n_layers=1, n=12000, seed=8)
    try:
        wl.step()
        torch.cuda.synchronize()
        out0, lse0 = wl.out.clone(), wl.lse.clone()
        ref = QC.oracle_unit(wl, 0, 0)
        cold = [int(t) for t in ref["tokens"] if ref["slot"][t] < 0][:100]
        assert len(cold) == 100
        staging = wl.cache.staging_ptr(0)
        base_row = (staging - wl.cache.pool.data_ptr()) // 2048
        toks = torch.tensor(cold, dtype=torch.int64, device="cuda")
        slots = torch.arange(base_row, base_row + len(cold), dtype=torch.int32, device="cuda")
        wl.cache.pool[slots.long()] = wl.host[0][0][toks.cpu()].cuda()
        wl.cache.slot_table_set(wl.handles[0], 0, toks, slots)
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        assert torch.equal(out0, wl.out) and torch.equal(lse0, wl.lse)
        # the slot table now holds the remapped rows
        h = wl.handles[0]
        assert torch.equal(wl.cache.slot_table[h.index, 0, toks], slots)
        QC.check_unit(wl, 0, 0)
    finally:
        wl.close()


def test_slot_table_fill_matches_oracle_layout():
    wl = workloads.build(2, [5000, 3000, 9000], [Q.KV_HBM, Q.KV_HOST_RING, Q.KV_HOST],
                         lambda l, r, n: synth.planted_uniform(n // 4, 10, r), staging_rows=16,
                         ring=1024, seed=9)
    try:
        torch.cuda.synchronize()
        for r in range(3):
            h = wl.handles[r]
            for l in range(2):
                got = wl.cache.slot_table[h.index, l, :wl.ctxs[r]].cpu().numpy()
                assert np.array_equal(got, QC.oracle_slot_row(wl, l, r)), (r, l)
    finally:
        wl.close()


def test_device_error_word_reports_bad_inputs():
    wl = workloads.tiny()
    try:
        h = wl.handles[0]
        # a slot outside the pool is refused and reported; the table keeps its value
        before = wl.cache.slot_table[h.index, 0, 5].item()
        wl.cache.slot_table_set(h, 0, torch.tensor([5], dtype=torch.int64, device="cuda"),
                                torch.tensor([1 << 30], dtype=torch.int32, device="cuda"))
        st, det = wl.cache.poll_error()
        assert st == Q.ERR_BAD_SLOT
        assert wl.cache.slot_table[h.index, 0, 5].item() == before
        assert wl.cache.poll_error()[0] == 0            # cleared by the read
        # a selected block outside the context is skipped and reported
        wl.step()
        wl.sel[0, 3] = 1 << 20
        wl.cache.sparse_decode_attn(wl.handles, 0, 1, wl.q, wl.sel, wl.nsel, wl.budget, None,
                                    wl.softmax_scale, wl.out, wl.lse)
        st, det = wl.cache.poll_error()
        assert st == Q.ERR_BAD_BLOCK and det == 1 << 20
        assert torch.isfinite(wl.out).all()
    finally:
        wl.close()


def test_stale_handle_rejected_by_compute_calls():
    wl = workloads.tiny()
    try:
        h = wl.handles[0]
        wl.cache.request_end(h)
        with pytest.raises(Q.QsaError) as e:
            wl.step()
        assert e.value.status == Q.ERR_STALE_HANDLE
        wl.handles[0] = wl.cache.request_begin(8192, Q.KV_HBM)
    finally:
        wl.close()


def test_c256k_x8_bench_configuration_sampled():
    """The benchmark's workload at full size: 8 requests x 12 layers x 262144
    tokens, host history + tail ring, layer-sequential calls exactly as
    bench.py makes them; sampled units checked against the oracle."""
    wl = workloads.c256k_x8()
    try:
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        for (l, r) in [(0, 0), (5, 3), (11, 7)]:
            res = QC.check_unit(wl, l, r)
            toks = res["ref"]["tokens"]
            hot = (res["ref"]["slot"][toks] >= 0).sum()
            assert 0.3 < hot / len(toks) < 0.7         # about half the rows from the HBM ring
    finally:
        wl.close()


def test_c1m_host_only_sampled():
    """1M-token contexts with KV only in pinned host memory (sinks + Zipf
    recency planting): 4 requests x 12 layers at full size (96 GiB of pinned
    host history), the captured two-micro-batch step as the benchmark runs
    it; sampled units from every request checked against the oracle."""
    wl = workloads.c1m_x4()
    try:
        g = wl.capture(2)
        g.replay()
        torch.cuda.synchronize()
        _clean(wl)
        for (l, r) in [(0, 0), (5, 1), (8, 2), (11, 3)]:
            res = QC.check_unit(wl, l, r)
            assert set(range(4)) <= set(res["ref"]["sel"].tolist())   # sink blocks kept
            assert (res["ref"]["slot"] == -1).all()                   # every row from host memory
        del g
    finally:
        wl.close()


def test_ragged_batch_recycling_on_gpu():
    """64 requests with log-uniform contexts in one batch per layer, all 12
    layers; 16 of them finish and 16 new requests are admitted in their slots
    under new generations with new contexts; every unit type is checked
    against the oracle before and after, and the cache counters return to
    their initial values at the end."""
    L = 12
    new_ctx = synth.log_uniform_contexts(16, 4096, 262144, seed=77)
    spare = sum(L * (n if n < 32768 else 4096) for n in new_ctx)   # room for the new leases
    wl = workloads.ragged(n_layers=L, extra_requests=0, spare_rows=spare)
    try:
        s0 = dict(wl.cache.stats())
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        R = wl.n_req
        hbm = [r for r in range(R) if wl.placements[r] == Q.KV_HBM]
        off = [r for r in range(R) if wl.placements[r] != Q.KV_HBM]
        assert hbm and off
        for r in hbm[:2] + off[:2]:
            QC.check_unit(wl, 11, r)
        rng = np.random.default_rng(3)
        done = [int(x) for x in rng.choice(R, 16, replace=False)]
        old = [wl.handles[r] for r in done]
        for j, r in enumerate(done):
            n = new_ctx[j]
            h = wl.reissue(r, n, Q.KV_HBM if n < 32768 else Q.KV_HOST_RING, seed=500 + j)
            assert h.generation == 2 and h.index == old[j].index
        for h in old:
            with pytest.raises(Q.QsaError) as e:
                wl.cache.request_info(h)
            assert e.value.status == Q.ERR_STALE_HANDLE
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        for i, r in enumerate(done[:4]):
            QC.check_unit(wl, 3 * i, r)
        for h in wl.handles:
            wl.cache.request_end(h)
        s_end = wl.cache.stats()
        assert s_end["active_requests"] == 0 and s_end["free_request_slots"] == R
        assert s_end["hbm_kv_bytes_in_use"] == 0
        assert s_end["free_hbm_rows"] == s0["hbm_pool_rows"] - s0["staging_rows_total"]
        assert s_end["free_ranges"] == 1
        wl.handles = []
    finally:
        wl.close()


def test_pipelined_graph_step_equals_sequential_step():
    """Request groups on separate streams, captured as a CUDA graph and
    replayed, give the same selections as the one-stream layer loop and the
    same attention to fp32 rounding (smaller calls spread a unit's splits
    over more CTAs, which changes only the merge order)."""
    wl = _host_ring_workload(n_req=4, n_layers=3, n=20000, seed=12)
    try:
        wl.step()
        torch.cuda.synchronize()
        ref = [t.clone() for t in (wl.sel, wl.nsel, wl.out, wl.lse)]
        for t in (wl.sel, wl.nsel, wl.out, wl.lse):
            t.zero_()
        g = wl.capture(2)
        for t in (wl.sel, wl.nsel, wl.out, wl.lse):
            t.zero_()
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        _clean(wl)
        assert torch.equal(ref[0], wl.sel) and torch.equal(ref[1], wl.nsel)
        assert torch.allclose(ref[2], wl.out, rtol=1e-5, atol=1e-6)
        assert torch.allclose(ref[3], wl.lse, rtol=1e-6, atol=1e-6)
        QC.check_unit(wl, 2, 3)
    finally:
        wl.close()


def test_index_score_work_counter_rearms_and_is_per_first_unit():
    """The index-score CTAs take tiles from a work counter that the call's
    last CTA re-arms.  Back-to-back calls, calls on two streams at once
    (different first units) and one call over several layers must all give
    the block scores of a single call, bit for bit (each score is computed
    by exactly one thread, whatever the schedule)."""
    ctxs = [70000, 9000, 130001, 4096]
    wl = workloads.build(
        3, ctxs, [Q.KV_HBM] * 4,
        lambda l, r, n: synth.planted_uniform(n // 4, 512, synth.mix_seed(31, 90, l, r)),
        staging_rows=64, seed=31)
    try:
        c, hs, R = wl.cache, wl.handles, wl.n_req
        wl.blk.fill_(7.0)       # entries past a unit's last block stay untouched
        c.index_score(hs, 0, 3, wl.q_idx, wl.w, wl.blk)
        torch.cuda.synchronize()
        ref = wl.blk.clone()
        for _ in range(4):
            wl.blk.fill_(7.0)
            c.index_score(hs, 0, 3, wl.q_idx, wl.w, wl.blk)
            torch.cuda.synchronize()
            assert torch.equal(ref, wl.blk)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        for l in range(3):
            sl = slice(l * R, (l + 1) * R)
            wl.blk[sl].fill_(7.0)
            s1.wait_stream(torch.cuda.current_stream())
            s2.wait_stream(torch.cuda.current_stream())
            for _ in range(3):
                wl.score_group_layer(0, 2, l, s1)
                wl.score_group_layer(2, 4, l, s2)
            torch.cuda.synchronize()
            assert torch.equal(ref[sl], wl.blk[sl])
        for l in range(3):
            wl.attn_group_layer(0, R, l, torch.cuda.current_stream())
        torch.cuda.synchronize()
        _clean(wl)
        for l in range(3):
            QC.check_unit(wl, l, 2)
            QC.check_unit(wl, l, 3)
    finally:
        wl.close()


def test_host_ring_on_host_numa_memory():
    """Host histories in qsa_host_alloc memory (host NUMA pages in the GPU's
    page tables): the decode step reads its cold rows there and matches the
    oracle, which reads the same bytes through the host mapping; freeing the
    memory of an ended request is accepted, a foreign pointer is refused."""
    wl = workloads.build(2, [20000] * 2, [Q.KV_HOST_RING] * 2,
                         lambda l, r, n: synth.planted_hot_cold(n // 4, 512, 1024,
                                                                synth.mix_seed(13, 90, l, r)),
                         seed=13, host_memory="vmm")
    try:
        assert getattr(wl.host[0], "_qsa_host_memory", None) is not None
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        for l in range(2):
            for r in range(2):
                res = QC.check_unit(wl, l, r)
                assert (res["ref"]["slot"][res["ref"]["tokens"]] == -1).any()   # some rows from host
    finally:
        wl.close()
    L = Q.lib()
    assert L.qsa_host_free(12345 * 4096) == Q.ERR_INVALID_ARG
