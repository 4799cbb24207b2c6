"""Parity of the FP8 KV variant (caches created with QSA_KV_FP8, 1040-byte rows)
with the fp64 oracle, through the C ABI.

Bars: selections bit-exact on a >= 1e-3 boundary gap; attention within 2e-3
of the oracle's attention over the same dequantised rows (the comparison is
against the FP8 values the cache holds, so the tolerance covers only the
kernel's arithmetic); gathered rows byte-exact; rows stored by
qsa_append_token bit-exact with oracle.quantize_kv_row_fp8.
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


def _fp8_ring_workload(n_req=2, n_layers=2, n=20000, seed=6):
    return workloads.build(n_layers, [n] * n_req, [Q.KV_HOST_RING] * n_req,
                           lambda l, r, n: synth.planted_hot_cold(n // 4, 512, 1024,
                                                                  synth.mix_seed(seed, 90, l, r)),
                           seed=seed, kv_format=Q.KV_FP8)


def test_fp8_cache_decode_step_gather_and_attention_modes():
    wl = _fp8_ring_workload()
    try:
        assert wl.cache.row_bytes == 1040 and wl.cache.pool.shape[1] == 1040
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        refs = {}
        for l in range(2):
            for r in range(2):
                refs[(l, r)] = QC.check_unit(wl, l, r)["ref"]
        out_direct, lse_direct = wl.out.clone(), wl.lse.clone()
        budget = wl.budget
        for l in range(2):
            sl = slice(l * 2, (l + 1) * 2)
            g = torch.empty(2, budget, 1040, dtype=torch.uint8, device="cuda")
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


def test_fp8_cache_hbm_requests_and_ragged_contexts():
    ctxs = [3, 1000, 2049, 6001]
    wl = workloads.build(1, ctxs, [Q.KV_HBM] * len(ctxs),
                         lambda l, r, n: synth.planted_uniform(n // 4, min(512, n // 4),
                                                               synth.mix_seed(8, 90, l, r)),
                         staging_rows=8, seed=8, kv_format=Q.KV_FP8)
    try:
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        for r in range(len(ctxs)):
            QC.check_unit(wl, 0, r)
    finally:
        wl.close()


def test_fp8_append_stores_quantised_rows_like_the_oracle():
    """Rows appended to an FP8 cache (HBM and host-ring requests) are the
    oracle's quantisation of the BF16 rows given, byte for byte, in the pool
    and in the host history."""
    n0, G, ring = 2000, 40, 512
    wl = workloads.build(1, [n0, n0], [Q.KV_HBM, Q.KV_HOST_RING], lambda l, r, n: [],
                         ring=ring, staging_rows=8, seed=9, grow=G, kv_format=Q.KV_FP8)
    try:
        c, hs, dev = wl.cache, wl.handles, wl.cache.pool.device
        g = torch.Generator().manual_seed(9)
        rows, keys = [], []
        for s in range(G):
            x = torch.randn(2, 1024, generator=g) * torch.exp2(torch.randint(-8, 8, (2, 1), generator=g).float())
            if s == 0:
                x[0, :128] = 0.0            # a zero head vector: scale 0, zero codes
                x[1, 128:256] = -0.0
            rows.append(x.to(torch.bfloat16).view(torch.uint8).view(2, 2048))
            keys.append(torch.randn(2, 64, generator=g))
            for h in hs:
                c.advance(h)
            c.append_token(hs, 0, 1, keys[s].to(dev), rows[s].to(dev))
        torch.cuda.synchronize()
        _clean(wl)
        info = [c.request_info(h) for h in hs]
        for s in range(G):
            t = n0 + s
            want = [O.quantize_kv_row_fp8(rows[s][r].numpy()) for r in range(2)]
            got_hbm = c.pool[info[0].hbm_row_base + t].cpu().numpy()
            assert np.array_equal(got_hbm, want[0]), s
            assert np.array_equal(wl.host[1][0, t].numpy(), want[1]), s
            ring_row = info[1].hbm_row_base + t % ring
            assert np.array_equal(c.pool[ring_row].cpu().numpy(), want[1]), s
            assert int(c.slot_table[hs[1].index, 0, t]) == ring_row
    finally:
        wl.close()


def test_fp8_many_host_units_in_one_launch():
    """32 host-ring units in one attention launch share the 64 host-reading
    CTAs: each CTA visits 64 splits, past the 32 whose row sources it
    resolves up front, so the later ones resolve as they are copied.  Plain,
    and with a hot cache planned into the attention over two steps (the
    second reads rows the first wrote back); every selected token's HBM row
    must hold its host row byte for byte, and the attention must match the
    oracle."""
    R, n = 32, 8200
    plant = lambda l, r, n: synth.planted_hot_cold(n // 4, 512, 1024, synth.mix_seed(9, 90, l, r))
    for hot in (0, 2048):
        wl = workloads.build(1, [n] * R, [Q.KV_HOST_RING] * R, plant, staging_rows=8, seed=9,
                             kv_format=Q.KV_FP8, hot_rows=hot)
        wl.fold_fill = hot > 0
        try:
            for _ in range(2 if hot else 1):
                wl.step()
                torch.cuda.synchronize()
                _clean(wl)
                for r in (0, 13, 31):
                    ref = QC.check_unit(wl, 0, r)["ref"]
                    toks = ref["tokens"]
                    h = wl.handles[r]
                    slots = wl.cache.slot_table[h.index, 0, :n].cpu().numpy()[toks]   # ring or hot rows
                    resident = slots >= 0
                    pool_rows = wl.cache.pool[torch.from_numpy(slots[resident].astype(np.int64)).cuda()]
                    host_rows = wl.host[r][0, torch.from_numpy(toks[resident].astype(np.int64))]
                    assert torch.equal(pool_rows.cpu(), host_rows), (hot, r)
        finally:
            wl.close()
