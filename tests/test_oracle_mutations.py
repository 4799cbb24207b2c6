"""Plant plausible slips in the oracle (on the CPU, in this process only) and
check that the pins in test_oracle_pins.py catch every one of them."""
import math

import numpy as np
import pytest

from oracle import qsa_oracle as O
from tests import test_oracle_pins as P


def _table(bias=7, subnormals=True):
    vals = []
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            vals.append(float("nan"))
        elif e == 0 and subnormals:
            vals.append(s * m / 8 * 2.0 ** (1 - bias))
        else:
            vals.append(s * (1 + m / 8) * 2.0 ** (e - bias))
    return np.array(vals)


def _scores_no_relu(codes, sc, q, w):
    k = O.decode_e4m3(codes) * O.decode_fp16(sc)[:, None]
    return (k @ np.asarray(q, float).T) @ np.asarray(w, float)


def _scores_no_scale(codes, sc, q, w):
    k = O.decode_e4m3(codes)
    return np.maximum(k @ np.asarray(q, float).T, 0) @ np.asarray(w, float)


def _scores_q_rows_swapped(codes, sc, q, w):
    k = O.decode_e4m3(codes) * O.decode_fp16(sc)[:, None]
    q = np.asarray(q, float)[::-1]
    return np.maximum(k @ q.T, 0) @ np.asarray(w, float)


def _blk_mean(S):
    S = np.asarray(S, float)
    return np.array([S[4 * b:4 * b + 4].mean() for b in range((len(S) + 3) // 4)])


def _blk_shifted(S):
    S = np.asarray(S, float)
    return np.array([S[max(0, 4 * b - 1):4 * b + 3].max() for b in range((len(S) + 3) // 4)])


def _select_tie_high(blk, budget):
    blk = np.asarray(blk, float)
    k = min(budget // 4, len(blk))
    order = np.lexsort((-np.arange(len(blk)), -blk))
    return np.sort(order[:k])


def _select_tokens_not_blocks(blk, budget):
    blk = np.asarray(blk, float)
    k = min(budget, len(blk))
    return np.sort(np.lexsort((np.arange(len(blk)), -blk))[:k])


def _select_unsorted(blk, budget):
    blk = np.asarray(blk, float)
    k = min(budget // 4, len(blk))
    return np.lexsort((np.arange(len(blk)), -blk))[:k]


def _tokens_unclipped(sel, n):
    return np.asarray([t for b in sel for t in range(4 * int(b), 4 * int(b) + 4)], dtype=np.int64)


def _ring_offset(ctx, layer, base, ring):
    t = np.arange(ctx)
    hot = t >= ctx - ring
    return np.where(hot, base + layer * ring + (t - (ctx - ring)), -1).astype(np.int32)


def _gather_host_only(tokens, slot, pool, host):
    return np.stack([host[int(t)] for t in tokens]) if len(tokens) else np.zeros((0, 2048), np.uint8)


def _attn_wrong_group(q_bits, rows, scale):
    q = O.decode_bf16(q_bits).reshape(16, 128)
    out = np.zeros((16, 128)); lse = np.full(16, -np.inf)
    if len(rows) == 0:
        return out, lse
    K, V = O.split_kv(rows)
    for h in range(16):
        g = h % 4
        lg = scale * (K[:, g] @ q[h]); m = lg.max(); p = np.exp(lg - m)
        out[h] = p @ V[:, g] / p.sum(); lse[h] = m + np.log(p.sum())
    return out, lse


def _attn_no_scale(q_bits, rows, scale):
    return O.__dict__["_orig_attn"](q_bits, rows, 1.0)


def _attn_lse_drops_max(q_bits, rows, scale):
    out, lse = O.__dict__["_orig_attn"](q_bits, rows, scale)
    if len(rows) == 0:
        return out, lse
    K, _ = O.split_kv(rows)
    q = O.decode_bf16(q_bits).reshape(16, 128)
    for h in range(16):
        lg = scale * (K[:, h // 4] @ q[h])
        lse[h] = np.log(np.exp(lg - lg.max()).sum())
    return out, lse


def _fp16_bias16(bits):
    return O.__dict__["_orig_fp16"](bits) * 0.5


def _bf16_drop_subnormal(bits):
    v = O.__dict__["_orig_bf16"](bits)
    b = np.asarray(bits, dtype=np.uint16)
    return np.where(((b >> 7) & 0xFF) == 0, 0.0, v)


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    pos = O.E4M3_POSITIVE
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    code = np.where(a - pos[lo] < pos[hi] - a, lo, hi).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def _encode_no_saturation(x):
    x = np.asarray(x, dtype=np.float64)
    code = O._orig_encode(x)
    return np.where(np.abs(x) > 448.0, code | np.uint8(0x7F), code).astype(np.uint8)


def _quantize_fp32_scale(k):
    k = np.asarray(k, dtype=np.float32).reshape(-1)
    q = np.float32(np.max(np.abs(k)) / np.float32(448.0))
    if q == 0:
        return np.zeros(k.size, dtype=np.uint8), 0
    x = np.clip((k / q).astype(np.float32), -448, 448)
    with np.errstate(over="ignore"):
        s16 = np.float16(q)
    return O.encode_e4m3(x), int(np.array(s16).view(np.uint16))


def _append_no_eviction(t, placement, base_row, layer, layer_rows, ring_tokens):
    w = O._orig_append(t, placement, base_row, layer, layer_rows, ring_tokens)
    return w[:1]


def _append_hbm_ring_stride(t, placement, base_row, layer, layer_rows, ring_tokens):
    if placement == "hbm":
        return [(t, base_row + layer * ring_tokens + t)]
    return O._orig_append(t, placement, base_row, layer, layer_rows, ring_tokens)


def _fp8_kv_swapped(rows_u8):
    K, V = O._orig_split_fp8(rows_u8)
    return V, K


def _fp8_one_scale(rows_u8):
    r = np.ascontiguousarray(rows_u8, dtype=np.uint8).reshape(-1, O.ROW_BYTES_FP8)
    kc = r[:, :512].reshape(-1, 4, 128)
    vc = r[:, 512:1024].reshape(-1, 4, 128)
    sc = np.ascontiguousarray(r[:, 1024:1040]).view(np.uint16).reshape(-1, 2, 4)
    ks = O.decode_fp16(sc[:, 0])
    return O.decode_e4m3(kc) * ks[:, :, None], O.decode_e4m3(vc) * ks[:, :, None]



def _hot_mutant(kind):
    """hot_cache_step with one slip (kind)."""
    def step(tokens, slot_row, owner, cursor, hot_base):
        slot = np.array(slot_row, dtype=np.int32, copy=True)
        own = np.array(owner, dtype=np.int32, copy=True)
        H = len(own)
        order = sorted(int(x) for x in tokens)
        if kind == "misses descending":
            order = order[::-1]
        in_use, misses = set(), []
        for t in order:
            s = int(slot[t])
            if hot_base <= s < hot_base + H:
                in_use.add(s - hot_base)
            elif s == -1:
                misses.append(t)
        if kind == "rows in use handed out":
            in_use = set()
        rows = [v for v in ((cursor + i) % H for i in range(H)) if v not in in_use][:len(misses)]
        fills = []
        for t, v in zip(misses, rows):
            e = int(own[v])
            if kind == "stale owner cleared":
                if e >= 0:
                    slot[e] = -1
            elif kind != "evicted token keeps its slot" and e >= 0 and int(slot[e]) == hot_base + v:
                slot[e] = -1
            own[v] = t
            slot[t] = hot_base + v
            fills.append((t, hot_base + v))
        if rows and kind != "cursor not advanced":
            cursor = rows[-1] if kind == "cursor on the last row" else (rows[-1] + 1) % H
        return slot, own, int(cursor), fills
    return step



def _gap_from_top(blk, budget_tokens):
    s = np.sort(np.asarray(blk, dtype=np.float64))[::-1]
    k = min(budget_tokens // 4, len(s))
    return float("inf") if k >= len(s) else float(s[0] - s[k])


def _gap_off_by_one(blk, budget_tokens):
    s = np.sort(np.asarray(blk, dtype=np.float64))[::-1]
    k = min(budget_tokens // 4, len(s))
    return float("inf") if k + 1 >= len(s) else float(s[k] - s[k + 1])



def _bf16_kv_swapped(rows_u8):
    k, v = O._orig_split_kv(rows_u8)
    return v, k


def _bf16_heads_interleaved(rows_u8):
    # K and V of each head side by side ([4][2][128]) instead of K[4][128] then V[4][128]
    bits = np.ascontiguousarray(rows_u8, dtype=np.uint8).view(np.uint16).reshape(-1, O.KV_HEADS, 2, O.HEAD_DIM)
    vals = O.decode_bf16(bits)
    return vals[:, :, 0, :], vals[:, :, 1, :]



def _resident_ctx_stride(ctx_len, layer, base_row, layer_rows=None):
    return (base_row + layer * ctx_len + np.arange(ctx_len, dtype=np.int64)).astype(np.int32)


def _resident_off_by_one(ctx_len, layer, base_row, layer_rows=None):
    stride = ctx_len if layer_rows is None else layer_rows
    return (base_row + layer * stride + 1 + np.arange(ctx_len, dtype=np.int64)).astype(np.int32)



def _layer_step_host_only(codes, scale_bits, q_idx, w, q_bits, slot_row, hbm_pool_rows, host_rows,
                          budget_tokens, softmax_scale):
    return O._orig_layer_step(codes, scale_bits, q_idx, w, q_bits, np.full_like(np.asarray(slot_row), -1),
                              hbm_pool_rows, host_rows, budget_tokens, softmax_scale)


MUTATIONS = {
    "unit step reads every row from the host history": {"layer_step": _layer_step_host_only},
    "resident slots with the context as layer stride": {"resident_slot_row": _resident_ctx_stride},
    "resident slots one row off": {"resident_slot_row": _resident_off_by_one},
    "bf16 row with K and V swapped": {"split_kv": _bf16_kv_swapped},
    "bf16 row with K and V interleaved per head": {"split_kv": _bf16_heads_interleaved},
    "boundary gap measured from the top block": {"boundary_gap": _gap_from_top},
    "boundary gap one place too low": {"boundary_gap": _gap_off_by_one},
    "hot cache: misses take rows in descending token order": {"hot_cache_step": _hot_mutant("misses descending")},
    "hot cache: rows in use by the step handed out": {"hot_cache_step": _hot_mutant("rows in use handed out")},
    "hot cache: evicted token keeps its slot": {"hot_cache_step": _hot_mutant("evicted token keeps its slot")},
    "hot cache: stale owner cleared": {"hot_cache_step": _hot_mutant("stale owner cleared")},
    "hot cache: cursor not advanced": {"hot_cache_step": _hot_mutant("cursor not advanced")},
    "hot cache: cursor left on the last row": {"hot_cache_step": _hot_mutant("cursor on the last row")},
    "fp8 row with K and V swapped": {"split_kv_fp8": _fp8_kv_swapped},
    "fp8 row with the K scales on V": {"split_kv_fp8": _fp8_one_scale},
    "e4m3 encoder ties away from zero": {"encode_e4m3": _encode_ties_away},
    "e4m3 encoder without saturation": {"encode_e4m3": _encode_no_saturation},
    "key scale not rounded to fp16": {"quantize_index_key": _quantize_fp32_scale},
    "ring append without eviction": {"append_slot_writes": _append_no_eviction},
    "resident append with the ring stride": {"append_slot_writes": _append_hbm_ring_stride},
    "e4m3 bias 8": {"E4M3_TABLE": _table(bias=8)},
    "e4m3 no subnormals": {"E4M3_TABLE": _table(subnormals=False)},
    "fp16 wrong bias": {"decode_fp16": _fp16_bias16},
    "bf16 subnormals flushed": {"decode_bf16": _bf16_drop_subnormal},
    "score without relu": {"token_scores": _scores_no_relu},
    "score without scale": {"token_scores": _scores_no_scale},
    "score with head rows swapped": {"token_scores": _scores_q_rows_swapped},
    "block mean instead of max": {"c4_block_scores": _blk_mean},
    "blocks shifted by one token": {"c4_block_scores": _blk_shifted},
    "tie rule reversed": {"select_blocks": _select_tie_high},
    "budget read as blocks": {"select_blocks": _select_tokens_not_blocks},
    "selection not sorted": {"select_blocks": _select_unsorted},
    "ragged tail not clipped": {"selected_tokens": _tokens_unclipped},
    "ring slot offset instead of modulo": {"ring_slot_row": _ring_offset},
    "gather ignores slot table": {"gather_rows": _gather_host_only},
    "GQA group h % 4": {"decode_attention": _attn_wrong_group},
    "softmax scale dropped": {"decode_attention": _attn_no_scale},
    "lse without the max term": {"decode_attention": _attn_lse_drops_max},
}


def _all_pins():
    pins = [getattr(P, n) for n in dir(P) if n.startswith("test_") and n != "test_c4_topk_hand_worked"]
    cases = P._load("c4_topk_hand.json")["cases"]
    pins += [(lambda c=c: P.test_c4_topk_hand_worked(c)) for c in cases]
    return pins


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    monkeypatch.setattr(O, "_orig_attn", O.decode_attention, raising=False)
    monkeypatch.setattr(O, "_orig_fp16", O.decode_fp16, raising=False)
    monkeypatch.setattr(O, "_orig_bf16", O.decode_bf16, raising=False)
    monkeypatch.setattr(O, "_orig_encode", O.encode_e4m3, raising=False)
    monkeypatch.setattr(O, "_orig_append", O.append_slot_writes, raising=False)
    monkeypatch.setattr(O, "_orig_split_fp8", O.split_kv_fp8, raising=False)
    monkeypatch.setattr(O, "_orig_split_kv", O.split_kv, raising=False)
    monkeypatch.setattr(O, "_orig_layer_step", O.layer_step, raising=False)
    for attr, val in MUTATIONS[name].items():
        monkeypatch.setattr(O, attr, val)
    caught = 0
    for pin in _all_pins():
        try:
            pin()
        except Exception:
            caught += 1
    assert caught > 0, f"no pin catches: {name}"
