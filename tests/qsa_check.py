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


# ------------------------------------------------ tight boundary gaps

TIGHT_GAP = (1.1e-3, 1.9e-3)   # fp64 boundary-gap window of the tight-gap tests
_ONE_FP16 = 0x3C00


def _fp16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def tune_boundary(codes, scale_bits, q_idx, w, budget, cand_codes, window=TIGHT_GAP,
                  margin=0.05):
    """Rewrite index keys of unselected blocks of one unit so that the
    oracle's fp64 boundary gap falls inside `window` (input construction for
    the tight-gap tests; the arithmetic is the oracle's):

      1. every unselected block within `margin` of the K-th best block score T
         gets the scales of its four tokens halved (exact for normal fp16)
         until it is not;
      2. the best unselected block b gets, in its first token, the codes of
         the first candidate row of cand_codes for which some fp16 scale puts
         that token's score in [T - window[1], T - window[0]], and that scale.
         Its other tokens are already at most T - margin, so the token's
         score is b's block score, and b is the best unselected block.

    The selected set does not change.  Returns (codes, scale_bits, b, token)
    as new arrays; raises AssertionError when no candidate fits."""
    codes = np.array(codes, dtype=np.uint8, copy=True)
    sb = np.array(scale_bits, dtype=np.uint16, copy=True)
    q_idx = np.asarray(q_idx, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    n = codes.shape[0]
    blk = O.c4_block_scores(O.token_scores(codes, sb, q_idx, w))
    nb = blk.shape[0]
    K = min(budget // 4, nb)
    assert K < nb, "every block is selected: there is no boundary"
    order = np.lexsort((np.arange(nb), -blk))
    sel0 = np.sort(order[:K])
    T = blk[order[K - 1]]
    assert T > margin + window[1], f"K-th best score {T} too small to place a gap below it"
    unsel = np.ones(nb, dtype=bool)
    unsel[sel0] = False

    def token_range(b):
        return np.arange(4 * b, min(n, 4 * b + 4))

    # 1. push every close unselected block below T - margin
    for _ in range(64):
        close = np.nonzero(unsel & (blk > T - margin))[0]
        if close.size == 0:
            break
        toks = np.concatenate([token_range(b) for b in close])
        sb[toks] = _fp16_bits(O.decode_fp16(sb[toks]) / 2.0)
        S = O.token_scores(codes[toks], sb[toks], q_idx, w)
        for b in close:
            m = (toks >= 4 * b) & (toks < 4 * b + 4)
            blk[b] = S[m].max()
    else:
        raise AssertionError("could not push the unselected blocks below the margin")

    # 2. the best unselected block takes a score just below T
    cand = np.nonzero(unsel)[0]
    b = int(cand[np.argmax(blk[cand])])
    t = 4 * b
    s8 = O.token_scores(cand_codes, np.full(cand_codes.shape[0], _ONE_FP16, dtype=np.uint16),
                        q_idx, w)
    lo_s, hi_s = T - window[1], T - window[0]
    for c in np.nonzero(s8 > 0)[0]:
        mid = np.float16(0.5 * (lo_s + hi_s) / s8[c]).view(np.uint16).astype(np.int64)
        hit = None
        for bits in (mid, mid - 1, mid + 1, mid - 2, mid + 2):
            if not (0 < bits < 0x7C00):
                continue
            s = O.decode_fp16(np.uint16(bits)) * s8[c]
            if lo_s <= s <= hi_s:
                hit = np.uint16(bits)
                break
        if hit is not None:
            codes[t] = cand_codes[c]
            sb[t] = hit
            break
    else:
        raise AssertionError("no candidate key reaches the gap window")

    blk2 = O.c4_block_scores(O.token_scores(codes, sb, q_idx, w))
    gap = O.boundary_gap(blk2, budget)
    assert window[0] <= gap <= window[1], gap
    assert np.array_equal(O.select_blocks(blk2, budget), sel0)
    return codes, sb, b, t
