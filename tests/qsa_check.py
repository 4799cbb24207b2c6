"""Test-side helpers: run the fp64 oracle on one decode unit of a workload and
compare with what the CUDA library produced.

Oracle inputs are the generator's bytes, read back from where the workload
builder placed them (index-key tensors, pool rows at the oracle's own slot
layout, pinned host rows); nothing the CUDA kernels wrote is fed to the
oracle.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import qsa_oracle as O
from sparse_attention_decode_qsa_gb300 import _native as N

ATTN_TOL = 2e-3          # max abs error of out and lse (bf16 inputs, fp32 accumulation)
SCORE_REL_TOL = 1e-5     # block-score error relative to sum_h w_h sc sum_d |q k|
MIN_GAP = 1e-3           # required fp64 score gap at the top-k boundary


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def unit_inputs(wl, l, r):
    h = wl.handles[r]
    n = wl.ctxs[r]
    u = wl.unit(l, r)
    codes = wl.cache.index_keys[h.index, l, :n].cpu().numpy()
    scales = bits16(wl.cache.index_scales[h.index, l, :n])
    return dict(n=n, codes=codes, scales=scales,
                q_idx=wl.q_idx[u].cpu().double().numpy(), w=wl.w[u].cpu().double().numpy(),
                q=bits16(wl.q[u]))


def oracle_slot_row(wl, l, r):
    info = wl.cache.request_info(wl.handles[r])
    n = wl.ctxs[r]
    p = wl.placements[r]
    if p == N.KV_HBM:
        return O.resident_slot_row(n, l, info.hbm_row_base, info.layer_rows)
    if p == N.KV_HOST_RING:
        return O.ring_slot_row(n, l, info.hbm_row_base, wl.cache.ring_tokens)
    return np.full(n, -1, dtype=np.int32)


class PoolRows:
    """Row accessor over the device pool for the few rows the oracle needs."""

    def __init__(self, pool: torch.Tensor, slots):
        slots = sorted(set(int(s) for s in slots if s >= 0))
        self.map = {}
        if slots:
            idx = torch.tensor(slots, dtype=torch.int64, device=pool.device)
            data = pool[idx].cpu().numpy()
            self.map = dict(zip(slots, data))

    def __getitem__(self, s):
        return self.map[int(s)]


def oracle_unit(wl, l, r, budget=None):
    """Run the oracle's steps on unit (l, r); returns the oracle's dict plus
    the per-block tolerance scale and the boundary gap."""
    budget = budget or wl.budget
    x = unit_inputs(wl, l, r)
    n = x["n"]
    S = O.token_scores(x["codes"], x["scales"], x["q_idx"], x["w"])
    blk = O.c4_block_scores(S)
    sel = O.select_blocks(blk, budget)
    toks = O.selected_tokens(sel, n)
    slot = oracle_slot_row(wl, l, r)
    pool = PoolRows(wl.cache.pool, slot[toks])
    host = wl.host[r][l, :n].numpy() if wl.host[r] is not None else None
    fp8 = wl.cache.kv_format == N.KV_FP8
    rows = O.gather_rows(toks, slot, pool, host, O.ROW_BYTES_FP8 if fp8 else O.ROW_BYTES)
    out, lse = O.decode_attention(x["q"], rows, wl.softmax_scale, "fp8" if fp8 else "bf16")
    # tolerance scale per token: sum_h w_h |sc| sum_d |q_hd e4m3(code_d)|
    absk = np.abs(O.decode_e4m3(x["codes"])) * np.abs(O.decode_fp16(x["scales"]))[:, None]
    mag = (absk @ np.abs(x["q_idx"]).T) @ np.abs(x["w"])
    mag_blk = O.c4_block_scores(mag)
    return dict(S=S, blk=blk, sel=sel, tokens=toks, rows=rows, out=out, lse=lse,
                mag_blk=mag_blk, gap=O.boundary_gap(blk, budget), slot=slot)


def check_unit(wl, l, r, ref=None, check_scores=True):
    """Compare the library's outputs of unit (l, r) with the oracle."""
    ref = ref or oracle_unit(wl, l, r)
    u = wl.unit(l, r)
    n = wl.ctxs[r]
    nb = (n + 3) // 4
    assert ref["gap"] >= MIN_GAP, f"unit ({l},{r}): boundary gap {ref['gap']} below {MIN_GAP}"
    if check_scores:
        g = wl.blk[u, :nb].cpu().double().numpy()
        err = np.abs(g - ref["blk"])
        bound = SCORE_REL_TOL * ref["mag_blk"] + 1e-30
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, f"unit ({l},{r}): {bad.size} block scores off, first {bad[:5]}"
    k = int(wl.nsel[u].item())
    assert k == len(ref["sel"])
    assert np.array_equal(wl.sel[u, :k].cpu().numpy(), ref["sel"]), f"unit ({l},{r}) selection"
    out = wl.out[u].cpu().double().numpy()
    lse = wl.lse[u].cpu().double().numpy()
    e_out = np.abs(out - ref["out"]).max()
    e_lse = np.abs(lse - ref["lse"]).max()
    assert e_out <= ATTN_TOL, f"unit ({l},{r}): attention max abs err {e_out}"
    assert e_lse <= ATTN_TOL, f"unit ({l},{r}): lse max abs err {e_lse}"
    return dict(err_out=e_out, err_lse=e_lse, ref=ref)
