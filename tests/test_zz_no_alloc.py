"""The no-allocation attention entry point, qsa_sparse_decode_attn_noalloc.

It serves callers that cannot allocate device memory where they run
attention (a pre-planned memory arena, a plug-in that only gets its input
and output buffers, code that must not trigger cudaMalloc's device
synchronisation).  This test calls it through the C ABI and compares it with
the existing entry point, qsa_sparse_decode_attn reading the same gathered
rows, on two calls in a row (different layers, so the second call finds the
first call's partials in the shared scratch array).  It also checks that
sizes beyond the stated limits are refused.

The file is named to be collected last, and it sets up everything itself, so
it passes alone in a fresh process as well as after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import sparse_attention_decode_qsa_gb300 as Q
from sparse_attention_decode_qsa_gb300 import _native as N
from sparse_attention_decode_qsa_gb300 import synth, workloads

pytestmark = pytest.mark.gpu

TOL = 2e-3   # the attention tolerance used by every parity test


def _call(q, rows, n_rows, n_units, stride, scale, out, lse):
    L = N.lib()
    return L.qsa_sparse_decode_attn_noalloc(
        q.view(torch.int16).data_ptr(), rows.data_ptr(), n_rows.data_ptr(), n_units, stride,
        C.c_float(scale), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_existing_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    seed = 21
    ctxs = [20000, 1001, 8192]
    wl = workloads.build(2, ctxs, [Q.KV_HOST_RING, Q.KV_HBM, Q.KV_HBM],
                         lambda l, r, n: synth.planted_hot_cold((n + 3) // 4, min(512, (n + 3) // 4),
                                                                1024, synth.mix_seed(seed, l, r)),
                         staging_rows=0, seed=seed)
    try:
        R, budget = wl.n_req, wl.budget
        for l in range(2):                           # two calls in a row
            sl = slice(l * R, (l + 1) * R)
            wl.step_layer(l)
            g = torch.empty(R, budget, 2048, dtype=torch.uint8, device="cuda")
            n_rows = torch.empty(R, dtype=torch.int32, device="cuda")
            wl.cache.gather_rows(wl.handles, l, 1, wl.sel[sl], wl.nsel[sl], budget, g, n_rows)
            ref_out = torch.empty(R, 16, 128, dtype=torch.float32, device="cuda")
            ref_lse = torch.empty(R, 16, dtype=torch.float32, device="cuda")
            wl.cache.sparse_decode_attn(wl.handles, l, 1, wl.q[sl], wl.sel[sl], wl.nsel[sl],
                                        budget, g, wl.softmax_scale, ref_out, ref_lse)
            out = torch.full((R, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
            lse = torch.full((R, 16), float("nan"), dtype=torch.float32, device="cuda")
            st = _call(wl.q[sl].contiguous(), g, n_rows, R, budget, wl.softmax_scale, out, lse)
            assert st == 0, N.lib().qsa_last_error_string()
            torch.cuda.synchronize()
            assert wl.cache.poll_error()[0] == 0
            assert torch.isfinite(out).all() and torch.isfinite(lse).all()
            assert (out - ref_out).abs().max().item() <= TOL
            assert (lse - ref_lse).abs().max().item() <= TOL
    finally:
        wl.close()


def test_noalloc_rejects_sizes_beyond_its_limits():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q = torch.zeros(17, 16, 128, dtype=torch.bfloat16, device="cuda")
    rows = torch.zeros(1, 16, 2048, dtype=torch.uint8, device="cuda")
    n_rows = torch.zeros(17, dtype=torch.int32, device="cuda")
    out = torch.zeros(17, 16, 128, dtype=torch.float32, device="cuda")
    lse = torch.zeros(17, 16, dtype=torch.float32, device="cuda")
    assert _call(q, rows, n_rows, N.STATIC_MAX_UNITS + 1, 16, 0.1, out, lse) == N.ERR_INVALID_ARG
    assert b"QSA_STATIC_MAX_UNITS" in N.lib().qsa_last_error_string()
    assert _call(q, rows, n_rows, 1, N.STATIC_MAX_ROWS + 4, 0.1, out, lse) == N.ERR_INVALID_ARG
    assert b"QSA_STATIC_MAX_ROWS" in N.lib().qsa_last_error_string()
    assert _call(q, rows, n_rows, 0, 16, 0.1, out, lse) == N.ERR_INVALID_ARG
