"""The no-allocation attention entry point, qsa_sparse_decode_attn_noalloc.

It serves callers that cannot allocate device memory where they run
attention (a pre-planned memory arena, a plug-in that only gets its input
and output buffers, code that must not trigger cudaMalloc's device
synchronisation).  This test calls it through the C ABI and compares it with
the existing entry point, qsa_sparse_decode_attn reading the same gathered
rows, and with the fp64 oracle's attention over the oracle's own gather of
the same tokens, on three calls in a row: two full-size calls (different
layers), then a call with only 100 rows per unit, so that partials the
full-size call left in the shared scratch array beyond the first 100 rows
would show if the merge read them.  It also checks that sizes beyond the
stated limits are refused.

The file is named to be collected last, and it sets up everything itself, so
it passes alone in a fresh process as well as after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import sparse_attention_decode_qsa_gb300 as Q
from oracle import qsa_oracle as O
from sparse_attention_decode_qsa_gb300 import _native as N
from sparse_attention_decode_qsa_gb300 import synth, workloads
from tests import qsa_check as QC

pytestmark = pytest.mark.gpu

TOL = 2e-3   # the attention tolerance used by every parity test


def _call(q, rows, n_rows, n_units, stride, scale, out, lse):
    L = N.lib()
    return L.qsa_sparse_decode_attn_noalloc(
        q.view(torch.int16).data_ptr(), rows.data_ptr(), n_rows.data_ptr(), n_units, stride,
        C.c_float(scale), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _close(out, lse, ref_out, ref_lse):
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    assert (out - ref_out).abs().max().item() <= TOL
    assert (lse - ref_lse).abs().max().item() <= TOL


def test_noalloc_matches_existing_entry_point_and_oracle_on_three_calls():
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
        small = 100                                   # rows per unit in the third call
        for call, l in enumerate([0, 1, 1]):
            sl = slice(l * R, (l + 1) * R)
            if call < 2:
                wl.step_layer(l)
            g = torch.empty(R, budget, 2048, dtype=torch.uint8, device="cuda")
            n_rows = torch.empty(R, dtype=torch.int32, device="cuda")
            wl.cache.gather_rows(wl.handles, l, 1, wl.sel[sl], wl.nsel[sl], budget, g, n_rows)
            nsel = wl.nsel[sl].clone()
            if call == 2:                             # the first small/4 selected blocks only
                nsel = torch.clamp(nsel, max=small // 4)
                n_rows = (4 * nsel).to(torch.int32)
            ref_out = torch.empty(R, 16, 128, dtype=torch.float32, device="cuda")
            ref_lse = torch.empty(R, 16, dtype=torch.float32, device="cuda")
            wl.cache.sparse_decode_attn(wl.handles, l, 1, wl.q[sl], wl.sel[sl], nsel, budget, g,
                                        wl.softmax_scale, ref_out, ref_lse)
            out = torch.full((R, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
            lse = torch.full((R, 16), float("nan"), dtype=torch.float32, device="cuda")
            st = _call(wl.q[sl].contiguous(), g, n_rows, R, budget, wl.softmax_scale, out, lse)
            assert st == 0, N.lib().qsa_last_error_string()
            torch.cuda.synchronize()
            assert wl.cache.poll_error()[0] == 0
            _close(out, lse, ref_out, ref_lse)
            # the oracle: its own gather of the unit's selected tokens (generator
            # bytes only), attention over the rows this call covers
            for r in range(R):
                ref = QC.oracle_unit(wl, l, r)
                m = int(n_rows[r].item())
                assert m == (min(small, len(ref["tokens"])) if call == 2 else len(ref["tokens"]))
                o_ref, lse_ref = O.decode_attention(QC.bits16(wl.q[wl.unit(l, r)]), ref["rows"][:m],
                                                    wl.softmax_scale)
                assert np.abs(out[r].cpu().double().numpy() - o_ref).max() <= TOL
                assert np.abs(lse[r].cpu().double().numpy() - lse_ref).max() <= TOL
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
