"""Pins that tie the fp64 oracle to facts outside itself.

Each test checks the oracle against something it does not compute: values
fixed by a format specification or worked by hand (tests/golden/), library
routines for special cases (numpy / torch decoders, torch's fp64 softmax
attention), closed forms, or invariants that any correct implementation must
satisfy.  They are chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand) makes one of them fail;
tests/test_oracle_mutations.py checks that claim by planting such slips.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from sparse_attention_decode_qsa_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- formats

def test_e4m3_spec_values():
    for code_s, val, _ in _load("e4m3_spec_values.json")["values"]:
        got = O.decode_e4m3(np.array([int(code_s, 16)], dtype=np.uint8))[0]
        if val == "nan":
            assert math.isnan(got), code_s
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code_s


def test_e4m3_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp16_matches_numpy_for_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = O.decode_fp16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_matches_torch_for_all_bit_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = O.decode_bf16(bits.numpy().view(np.uint16))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------------- index score

def _hand_score_inputs():
    codes = np.zeros((6, 64), dtype=np.uint8)
    codes[0, :] = 0x38
    codes[1, :] = 0xB8
    codes[2, 0] = 0x40
    codes[3, :] = 0x7E
    codes[4, :] = 0x01
    codes[5, :32] = 0x7E
    codes[5, 32:] = 0xFE
    scales = np.array([0x3C00, 0x3C00, 0x3800, 0x0000, 0x4400, 0x2000], dtype=np.uint16)
    q = np.zeros((8, 64))
    q[0, :] = 1.0
    q[1, :] = -1.0
    q[2, 0] = 2.0
    g = _load("index_score_hand.json")
    w = np.array(g["w"])
    return codes, scales, q, w, g


def test_index_score_hand_worked():
    codes, scales, q, w, g = _hand_score_inputs()
    S = O.token_scores(codes, scales, q, w)
    assert S.tolist() == [t["S"] for t in g["tokens"]]
    assert O.c4_block_scores(S).tolist() == g["blocks"]["scores"]


def test_index_score_one_hot_picks_single_element():
    """q = e_d in head h only, w = e_h: S_t = relu(scale_t * e4m3(code[t][d])).
    Checked against torch's fp8 decoding and numpy's fp16 decoding, for every
    (h, d) on a few positions, which pins the index order of q, w and keys."""
    rng = np.random.default_rng(7)
    n = 32
    codes = rng.integers(0, 256, size=(n, 64), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30          # no NaN codes
    scales = (rng.random(n) * 4).astype(np.float16).view(np.uint16)
    ref_k = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * \
        scales.view(np.float16).astype(np.float64)[:, None]
    for h in (0, 3, 7):
        for d in (0, 1, 17, 63):
            q = np.zeros((8, 64)); q[h, d] = 1.0
            w = np.zeros(8); w[h] = 1.0
            S = O.token_scores(codes, scales, q, w)
            assert np.array_equal(S, np.maximum(ref_k[:, d], 0.0))


def test_index_score_invariants():
    u = synth.unit_inputs(256, seed=11, planted_blocks=[], device="cpu")
    codes = u.codes.numpy(); sc = u.scales.view(torch.int16).numpy().view(np.uint16)
    q = u.q_idx.double().numpy(); w = u.w.double().numpy()
    S = O.token_scores(codes, sc, q, w)
    assert (S >= 0).all()
    # linear in w (c > 0), and positively homogeneous in q
    assert np.allclose(O.token_scores(codes, sc, q, 3.0 * w), 3.0 * S, rtol=1e-14, atol=0)
    assert np.allclose(O.token_scores(codes, sc, 2.0 * q, w), 2.0 * S, rtol=1e-14, atol=0)
    # permuting tokens permutes scores
    p = np.random.default_rng(3).permutation(256)
    assert np.array_equal(O.token_scores(codes[p], sc[p], q, w), S[p])
    # zero scale -> zero score
    sc0 = sc.copy(); sc0[5] = 0
    assert O.token_scores(codes, sc0, q, w)[5] == 0.0
    # relu: negating every key of a token swaps which heads contribute
    neg = codes.copy(); neg[9] ^= 0x80
    a = O.token_scores(codes[9:10], sc[9:10], q, w)[0]
    b = O.token_scores(neg[9:10], sc[9:10], q, w)[0]
    k = O.decode_e4m3(codes[9]) * O.decode_fp16(sc[9:10])[0]
    dots = q @ k
    assert np.isclose(a, (np.maximum(dots, 0) * w).sum(), rtol=1e-14)
    assert np.isclose(b, (np.maximum(-dots, 0) * w).sum(), rtol=1e-14)
    assert np.isclose(a - b, (dots * w).sum(), rtol=1e-12)   # relu(x) - relu(-x) = x


# ----------------------------------------------------------- C4 and top-k

@pytest.mark.parametrize("case", _load("c4_topk_hand.json")["cases"], ids=lambda c: c["name"])
def test_c4_topk_hand_worked(case):
    blk = O.c4_block_scores(np.array(case["token_scores"], dtype=np.float64))
    assert blk.tolist() == case["blocks"]
    assert O.select_blocks(blk, case["budget"]).tolist() == case["selected"]


def _is_top_k(blk, sel, k):
    """Definition of the selection: |sel| = k, and every selected block ranks
    strictly above every unselected one under (score desc, id asc)."""
    sel = set(int(b) for b in sel)
    if len(sel) != k:
        return False
    rank = lambda b: (-blk[b], b)
    worst_in = max(rank(b) for b in sel)
    return all(rank(b) > worst_in for b in range(len(blk)) if b not in sel)


def test_topk_definition_on_random_inputs_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(200):
        nb = int(rng.integers(1, 300))
        blk = rng.integers(0, 6, size=nb).astype(np.float64)   # many ties
        budget = 4 * int(rng.integers(1, 80))
        sel = O.select_blocks(blk, budget)
        k = min(budget // 4, nb)
        assert list(sel) == sorted(sel)
        assert _is_top_k(blk, sel, k)


def test_topk_permutation_invariance():
    rng = np.random.default_rng(9)
    blk = rng.standard_normal(1000)
    sel = set(O.select_blocks(blk, 400).tolist())
    p = rng.permutation(1000)          # new block i holds old block p[i]
    sel_p = O.select_blocks(blk[p], 400)
    assert set(int(p[i]) for i in sel_p) == sel


def test_planted_set_is_selected():
    """A config-0 sized unit: the 512 planted blocks are exactly the top 512,
    with a boundary gap far above 1e-3."""
    n = 8192
    planted = synth.planted_uniform(n // 4, 512, seed=1)
    u = synth.unit_inputs(n, seed=2, planted_blocks=planted, device="cpu")
    S = O.token_scores(u.codes.numpy(), u.scales.view(torch.int16).numpy().view(np.uint16),
                       u.q_idx.numpy(), u.w.numpy())
    blk = O.c4_block_scores(S)
    sel = O.select_blocks(blk, 2048)
    assert sel.tolist() == planted.tolist()
    assert O.boundary_gap(blk, 2048) > 1.0


def test_selected_tokens_ragged_tail():
    assert O.selected_tokens([0, 2], 10).tolist() == [0, 1, 2, 3, 8, 9]
    assert O.selected_tokens([], 10).tolist() == []


# --------------------------------------------------------- slot table

def test_ring_slot_row_hand_worked():
    g = _load("ring_slots_hand.json")
    got = O.ring_slot_row(g["ctx_len"], g["layer"], g["base_row"], g["ring_tokens"])
    assert got.tolist() == g["slots"]


def test_gather_through_remapped_slots_is_identical():
    rng = np.random.default_rng(1)
    n = 64
    host = rng.integers(0, 256, size=(n, 2048), dtype=np.uint8)
    pool = np.zeros((200, 2048), dtype=np.uint8)
    slot = np.full(n, -1, dtype=np.int32)
    # move a few tokens into arbitrary pool rows holding the same bytes
    for t, s in [(3, 17), (40, 199), (63, 0), (10, 5)]:
        pool[s] = host[t]
        slot[t] = s
    toks = np.arange(n)
    a = O.gather_rows(toks, slot, pool, host)
    assert np.array_equal(a, host)
    # a slot pointing at a row with other bytes is visible
    slot[3] = 1
    assert not np.array_equal(O.gather_rows(toks, slot, pool, host), host)


# ---------------------------------------------------------- attention

def _rows_from(K, V):
    """Pack float K, V [m][4][128] as bf16 rows (K then V)."""
    kb = torch.from_numpy(K).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    vb = torch.from_numpy(V).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return np.concatenate([kb.reshape(len(K), -1), vb.reshape(len(V), -1)], axis=1).view(np.uint8)


def _q_bits(q):
    return torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_attention_dense_matches_torch_sdpa():
    """Budget >= context: the whole path is dense attention, which torch's
    fp64 scaled_dot_product_attention computes independently (GQA expanded by
    repeating each KV head for its 4 query heads)."""
    n = 37
    u = synth.unit_inputs(n, seed=4, planted_blocks=[], device="cpu")
    rows = synth.kv_rows(n, seed=5).numpy()
    qb = u.q.view(torch.int16).numpy().view(np.uint16)
    slot = np.full(n, -1, dtype=np.int32)
    res = O.layer_step(u.codes.numpy(), u.scales.view(torch.int16).numpy().view(np.uint16),
                       u.q_idx.numpy(), u.w.numpy(), qb, slot, None, rows, 2048, 1 / math.sqrt(128))
    assert res["tokens"].tolist() == list(range(n))
    rt = torch.from_numpy(rows).view(torch.bfloat16).reshape(n, 2, 4, 128).double()
    K = rt[:, 0].permute(1, 0, 2).repeat_interleave(4, dim=0)      # [16][n][128]
    V = rt[:, 1].permute(1, 0, 2).repeat_interleave(4, dim=0)
    q = u.q.double().reshape(16, 1, 128)
    ref = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=1 / math.sqrt(128))
    assert np.allclose(res["out"], ref.reshape(16, 128).numpy(), rtol=0, atol=1e-12)
    logits = torch.einsum("hd,hnd->hn", u.q.double(), K) / math.sqrt(128)
    assert np.allclose(res["lse"], torch.logsumexp(logits, dim=1).numpy(), rtol=0, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((16, 128))
    # one row: output = V, lse = its logit
    K = rng.standard_normal((1, 4, 128)); V = rng.standard_normal((1, 4, 128))
    rows = _rows_from(K, V)
    Kd, Vd = O.split_kv(rows)
    out, lse = O.decode_attention(_q_bits(q), rows, 0.5)
    qd = O.decode_bf16(_q_bits(q))
    for h in range(16):
        assert np.array_equal(out[h], Vd[0, h // 4])
        assert np.isclose(lse[h], 0.5 * qd[h] @ Kd[0, h // 4], rtol=1e-15)
    # identical keys: uniform weights, output = mean of V, lse = logit + log m
    m = 9
    K = np.repeat(rng.standard_normal((1, 4, 128)), m, axis=0)
    V = rng.standard_normal((m, 4, 128))
    rows = _rows_from(K, V)
    Kd, Vd = O.split_kv(rows)
    out, lse = O.decode_attention(_q_bits(q), rows, 0.25)
    for h in range(16):
        g = h // 4
        assert np.allclose(out[h], Vd[:, g].mean(axis=0), rtol=0, atol=1e-13)
        assert np.isclose(lse[h], 0.25 * qd[h] @ Kd[0, g] + math.log(m), rtol=1e-14)
    # no rows: zeros and -inf
    out, lse = O.decode_attention(_q_bits(q), np.zeros((0, 2048), np.uint8), 0.25)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_attention_split_merge_and_permutation():
    """Attention over A u B equals the log-sum-exp merge of A and B
    (o = (e^{lse_A} o_A + e^{lse_B} o_B) / (e^{lse_A} + e^{lse_B}),
    lse = log(e^{lse_A} + e^{lse_B})), and row order does not matter."""
    rng = np.random.default_rng(8)
    rows = synth.kv_rows(50, seed=9).numpy()
    qb = _q_bits(rng.standard_normal((16, 128)))
    o, l = O.decode_attention(qb, rows, 0.1)
    oa, la = O.decode_attention(qb, rows[:20], 0.1)
    ob, lb = O.decode_attention(qb, rows[20:], 0.1)
    M = np.maximum(la, lb)
    wa, wb = np.exp(la - M), np.exp(lb - M)
    om = (wa[:, None] * oa + wb[:, None] * ob) / (wa + wb)[:, None]
    assert np.allclose(o, om, rtol=0, atol=1e-13)
    assert np.allclose(l, M + np.log(wa + wb), rtol=0, atol=1e-13)
    p = rng.permutation(50)
    op, lp = O.decode_attention(qb, rows[p], 0.1)
    assert np.allclose(o, op, rtol=0, atol=1e-13) and np.allclose(l, lp, rtol=0, atol=1e-13)


def test_gqa_grouping_uses_contiguous_heads():
    """Changing KV head g's keys moves only query heads 4g..4g+3."""
    rows = synth.kv_rows(12, seed=3).numpy().copy()
    qb = _q_bits(np.random.default_rng(0).standard_normal((16, 128)))
    o1, _ = O.decode_attention(qb, rows, 0.1)
    r2 = rows.copy().view(np.uint16).reshape(12, 2, 4, 128)
    r2[:, 0, 2, :] ^= 0x8000                 # flip the sign of K of KV head 2
    o2, _ = O.decode_attention(qb, r2.reshape(12, -1).view(np.uint8), 0.1)
    changed = [h for h in range(16) if not np.array_equal(o1[h], o2[h])]
    assert changed == [8, 9, 10, 11]


# ------------------------------------------------------ byte accounting

def test_page_byte_accounting():
    g = _load("page_sizes.json")
    assert O.ROW_BYTES == g["kv_bytes_per_token_per_layer"]["value"]
    assert O.INDEX_DIM + 2 == g["index_key_bytes_per_token_per_layer"]["value"]
    n = 262144
    blk = np.arange(n // 4, dtype=np.float64)
    toks = O.selected_tokens(O.select_blocks(blk, g["indexer_budget_tokens"]["value"]), n)
    assert len(toks) == g["indexer_budget_tokens"]["value"]
    assert len(toks) * O.ROW_BYTES * g["qsa_layers"]["value"] == g["bytes_moved_per_decode_step"]["value"]
    assert 4 * len(O.select_blocks(blk, 2048)) == 2048 and g["c4_block_tokens"]["value"] == 4


# ---------------------------------------------------- producer side: append

def test_encode_e4m3_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = O.decode_e4m3(codes)
    vals = np.where(codes == 0x80, -0.0, vals)          # the decoder returns -0.0 as 0.0 * -1
    assert np.array_equal(O.encode_e4m3(vals), codes)


def test_encode_e4m3_nearest_ties_to_even_and_saturation():
    pos = O.E4M3_POSITIVE
    mid = (pos[:-1] + pos[1:]) / 2
    lo_codes = np.arange(0x7E, dtype=np.uint8)
    even = np.where(lo_codes % 2 == 0, lo_codes, lo_codes + 1).astype(np.uint8)
    assert np.array_equal(O.encode_e4m3(mid), even)
    assert np.array_equal(O.encode_e4m3(-mid), even | 0x80)
    step = (pos[1:] - pos[:-1]) * 1e-3
    assert np.array_equal(O.encode_e4m3(mid - step), lo_codes)
    assert np.array_equal(O.encode_e4m3(mid + step), lo_codes + 1)
    assert list(O.encode_e4m3([448.0, 449.0, 464.0, 1e30, -500.0])) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_encode_e4m3_matches_torch_on_in_range_values():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000),
                        rng.standard_normal(2000) * 1e-3, (O.E4M3_POSITIVE[:-1] + O.E4M3_POSITIVE[1:]) / 2])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.encode_e4m3(x), ref)


def test_quantize_index_key_hand_worked():
    cases = _load("quantize_hand.json")["cases"]
    for c in cases:
        k = np.zeros(64, dtype=np.float32)
        for d, v in c["nonzero"]:
            k[d] = v
        codes, sbits = O.quantize_index_key(k)
        want = np.zeros(64, dtype=np.uint8)
        for d, code in c["codes"]:
            want[d] = int(code, 16)
        assert sbits == int(c["scale_bits"], 16), c["why"]
        assert np.array_equal(codes, want), c["why"]


def test_quantize_index_key_matches_the_input_generator():
    """The generator's torch rounding (fp16 scale, float8_e4m3fn codes) and
    the oracle's own encoders agree on random keys of every magnitude."""
    rng = np.random.default_rng(9)
    keys = rng.standard_normal((300, 64)).astype(np.float32)
    keys *= np.exp2(rng.integers(-20, 20, size=(300, 1))).astype(np.float32)
    keys[0] = 0.0
    kt = torch.from_numpy(keys)
    sc = (kt.abs().amax(dim=1) / 448.0).to(torch.float16)
    x = (kt / torch.where(sc.float() > 0, sc.float(), torch.ones(300))[:, None]).clamp(-448, 448)
    x = torch.where((sc.float() > 0)[:, None], x, torch.zeros_like(x))
    ref_codes = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref_bits = sc.view(torch.int16).numpy().view(np.uint16)
    for i in range(300):
        codes, sbits = O.quantize_index_key(keys[i])
        assert sbits == int(ref_bits[i])
        assert np.array_equal(codes, ref_codes[i]), i


def test_append_slot_writes_reproduce_the_ring_and_resident_layouts():
    ring, base = 16, 100
    for layer in (0, 2):
        row = list(O.ring_slot_row(5, layer, base, ring)) + [-1] * 60
        for t in range(5, 60):
            for tok, s in O.append_slot_writes(t, "ring", base, layer, 0, ring):
                row[tok] = s
        assert np.array_equal(np.array(row[:60]), O.ring_slot_row(60, layer, base, ring))
    cap = 80
    row = [-1] * cap
    for t in range(cap):
        for tok, s in O.append_slot_writes(t, "hbm", base, 3, cap, ring):
            row[tok] = s
    assert row == [base + 3 * cap + t for t in range(cap)]
    assert O.append_slot_writes(7, "host", base, 1, 0, ring) == [(7, -1)]
    # hand-worked: ring of 4 at base 10, layer 1; token 9 takes ring row 10+4+1 and evicts token 5
    assert O.append_slot_writes(9, "ring", 10, 1, 0, 4) == [(9, 15), (5, -1)]


# ------------------------------------------------------------- FP8 KV rows

def _bf16_bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_fp8_row_decode_hand_worked():
    """Layout: K codes [4][128] at 0, V codes [4][128] at 512, fp16 scales
    K[0..3] at 1024, V[0..3] at 1032."""
    row = np.zeros(1040, dtype=np.uint8)
    sc = np.zeros(8, dtype=np.uint16)
    row[0 * 128 + 0] = 0x38            # K head 0 dim 0: 1.0 ...
    sc[0] = 0x3C00                     # ... times scale 1.0 = 1.0
    row[2 * 128 + 5] = 0x7E            # K head 2 dim 5: 448 ...
    sc[2] = 0x2000                     # ... times 2^-7 = 3.5
    row[512 + 1 * 128 + 127] = 0xB8    # V head 1 dim 127: -1.0 ...
    sc[4 + 1] = 0x4000                 # ... times 2.0 = -2.0
    row[512 + 3 * 128 + 64] = 0x01     # V head 3 dim 64: 2^-9 ...
    sc[4 + 3] = 0x7BFF                 # ... times 65504 = 127.9375
    row[1024:1040] = sc.view(np.uint8)
    K, V = O.split_kv_fp8(row[None])
    assert K.shape == (1, 4, 128) and V.shape == (1, 4, 128)
    want_k = np.zeros((4, 128)); want_k[0, 0] = 1.0; want_k[2, 5] = 3.5
    want_v = np.zeros((4, 128)); want_v[1, 127] = -2.0; want_v[3, 64] = 127.9375
    assert np.array_equal(K[0], want_k) and np.array_equal(V[0], want_v)


def test_fp8_row_quantize_hand_worked():
    k = np.zeros((4, 128), dtype=np.float32)
    v = np.zeros((4, 128), dtype=np.float32)
    k[1, 0], k[1, 1], k[1, 2] = 448.0, 1.0625, -1.1875     # scale 1.0: 0x7E, tie -> 0x38, tie -> 0xBA
    v[3, 0], v[3, 1] = -3.5, 1.75                         # scale 2^-7: -448 -> 0xFE, 224 -> 0x76
    row = np.concatenate([_bf16_bits(k.reshape(-1)), _bf16_bits(v.reshape(-1))]).view(np.uint8)
    f = O.quantize_kv_row_fp8(row)
    codes, scales = f[:1024], f[1024:].view(np.uint16)
    assert list(scales) == [0, 0x3C00, 0, 0, 0, 0, 0, 0x2000]
    assert list(codes[128:131]) == [0x7E, 0x38, 0xBA]
    assert list(codes[512 + 384:512 + 386]) == [0xFE, 0x76]
    assert np.count_nonzero(codes) == 5


def test_fp8_row_quantize_matches_torch_rounding_and_bound():
    rng = np.random.default_rng(11)
    for _ in range(40):
        x = torch.from_numpy(rng.standard_normal(1024).astype(np.float32) *
                             np.float32(2.0 ** rng.integers(-12, 12)))
        bf = x.to(torch.bfloat16)
        row = bf.view(torch.int16).numpy().view(np.uint8)
        f = O.quantize_kv_row_fp8(row)
        v = bf.float().view(8, 128)
        sc = (v.abs().amax(dim=1) / 448.0).to(torch.float16)
        q = (v / torch.where(sc.float() > 0, sc.float(), torch.ones(8))[:, None]).clamp(-448, 448)
        ref_codes = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(-1)
        assert np.array_equal(f[:1024], ref_codes)
        assert np.array_equal(f[1024:].view(np.uint16), sc.view(torch.int16).numpy().view(np.uint16))
        K, V = O.split_kv(row[None])
        Kq, Vq = O.split_kv_fp8(f[None])
        vals = np.concatenate([K, V], axis=1)[0]
        deq = np.concatenate([Kq, Vq], axis=1)[0]
        scale = O.decode_fp16(f[1024:].view(np.uint16))[:, None]
        # E4M3 round-to-nearest: half a step of 2^-3 relative, or of 2^-9 * scale below 2^-6
        assert np.all(np.abs(deq - vals) <= np.maximum(np.abs(vals) * 2.0 ** -4, scale * 2.0 ** -10) + 1e-30)


def test_fp8_attention_matches_torch_sdpa_on_dequantised_rows():
    rng = np.random.default_rng(12)
    m = 37
    rows = np.stack([O.quantize_kv_row_fp8(
        torch.from_numpy(rng.standard_normal(1024).astype(np.float32)).to(torch.bfloat16)
        .view(torch.int16).numpy().view(np.uint8)) for _ in range(m)])
    qb = torch.randn(16, 128).to(torch.bfloat16)
    out, lse = O.decode_attention(qb.view(torch.int16).numpy().view(np.uint16), rows, 0.1, "fp8")
    K, V = O.split_kv_fp8(rows)
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(4, dim=0)      # [16][m][128]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(4, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qb.double()[:, None, :], kt, vt, scale=0.1)
    assert np.abs(out - ref[:, 0].numpy()).max() < 1e-12
    logits = 0.1 * torch.einsum("hd,hmd->hm", qb.double(), kt)
    assert np.abs(lse - torch.logsumexp(logits, dim=1).numpy()).max() < 1e-12


# ------------------------------------------------ cross-step hot cache

def test_hot_cache_hand_worked():
    """Seven steps worked out by hand: cold start, hits and evictions, a
    returning token, the circular walk skipping a row in use, an all-hit step,
    a stale owner after a remap, and more misses than free rows."""
    g = _load("hot_cache_hand.json")
    slot = np.array(g["initial_slots"], dtype=np.int32)
    own = np.full(g["hot_rows"], -1, dtype=np.int32)
    cur = 0
    for i, st in enumerate(g["steps"]):
        for t, s in st.get("remap", []):
            slot[t] = s
        slot, own, cur, fills = O.hot_cache_step(st["tokens"], slot, own, cur, g["hot_base"])
        assert slot.tolist() == st["slots"], (i, st["note"])
        assert own.tolist() == st["owner"], (i, st["note"])
        assert cur == st["cursor"], (i, st["note"])
        assert [list(f) for f in fills] == st["fills"], (i, st["note"])


def test_hot_cache_invariants_on_drifting_selections():
    """Random selections that drift step to step (some steps keep everything,
    some redraw everything), with tail-ring tokens among them: after every
    step each selected token has a pool slot, hits and ring tokens keep
    theirs, exactly the selected cold tokens are filled, into distinct hot
    rows, which are the free rows nearest the cursor in circular order; other
    tokens only lose hot rows; the owner array and the slot table agree; and
    a gather through the new slot table returns the host bytes."""
    rng = np.random.default_rng(11)
    n, ring, H, base, ring_base, k = 400, 32, 48, 1000, 5000, 40
    host = rng.integers(0, 256, (n, 16), dtype=np.uint8)
    slot = np.full(n, -1, dtype=np.int32)
    pool = {}
    for t in range(n - ring, n):
        slot[t] = ring_base + t % ring
        pool[int(slot[t])] = host[t]
    own = np.full(H, -1, dtype=np.int32)
    cur = 0
    sel = np.sort(rng.choice(n, k, replace=False))
    for step in range(80):
        churn = [0.0, 0.1, 0.5, 1.0][step % 4]
        keep = sel[rng.random(k) >= churn]
        fresh = rng.permutation(np.setdiff1d(np.arange(n), keep))[:k - len(keep)]
        sel = np.sort(np.concatenate([keep, fresh]))
        before = slot.copy()
        slot, own, new_cur, fills = O.hot_cache_step(sel, slot, own, cur, base)
        for t, r in fills:
            pool[r] = host[t]
        in_sel = set(sel.tolist())
        assert all(slot[t] >= 0 for t in sel)
        assert all(slot[t] == before[t] for t in sel if before[t] >= 0)
        assert [t for t, _ in fills] == [t for t in sel if before[t] == -1]
        rows = [r - base for _, r in fills]
        assert all(0 <= v < H for v in rows) and len(set(rows)) == len(rows)
        in_use = {int(before[t]) - base for t in sel if base <= before[t] < base + H}
        nearest = sorted((v for v in range(H) if v not in in_use), key=lambda v: (v - cur) % H)
        assert rows == nearest[:len(rows)]
        if rows:
            assert new_cur == (rows[-1] + 1) % H
        else:
            assert new_cur == cur
        for t in range(n):
            if t not in in_sel and slot[t] != before[t]:
                assert slot[t] == -1 and base <= before[t] < base + H
        hot = [t for t in range(n) if base <= slot[t] < base + H]
        assert len({int(slot[t]) for t in hot}) == len(hot)
        assert all(own[slot[t] - base] == t for t in hot)
        assert np.array_equal(O.gather_rows(sel, slot, pool, host, row_bytes=16), host[sel])
        cur = new_cur


def test_boundary_gap_hand_worked():
    """The fp64 gap between the K-th best block score and the (K+1)-th, the
    quantity the parity tests require to be >= 1e-3 before they compare
    selections bit for bit; worked out by hand."""
    blk = [5.0, 1.0, 3.0, 9.0, 7.0, 2.0]                 # sorted: 9 7 5 3 2 1
    assert O.boundary_gap(blk, 12) == 2.0                 # K = 3: 5 - 3
    assert O.boundary_gap(blk, 10) == 2.0                 # K = 2 (10 tokens = 2 whole blocks): 7 - 5
    assert O.boundary_gap(blk, 4) == 2.0                  # K = 1: 9 - 7
    assert O.boundary_gap(blk, 20) == 1.0                 # K = 5: 2 - 1
    assert O.boundary_gap([4.0, 4.0, 4.0, 1.0], 8) == 0.0  # a tie at the boundary
    assert O.boundary_gap([1.0, 2.0], 8) == float("inf")  # every block selected
    assert O.boundary_gap([-1.0, -5.0, -2.0], 4) == 1.0   # K = 1: -1 - (-2)


def test_resident_slot_row_hand_worked():
    """An HBM-resident request's slot row: token t of layer l sits in pool row
    base + l * layer_rows + t, where layer_rows is the region's rows per
    layer (the request's capacity), and the context length when none is
    given; worked out by hand."""
    assert O.resident_slot_row(5, 2, 100, 8).tolist() == [116, 117, 118, 119, 120]
    assert O.resident_slot_row(3, 0, 7).tolist() == [7, 8, 9]
    assert O.resident_slot_row(3, 1, 7).tolist() == [10, 11, 12]
    assert O.resident_slot_row(4, 3, 0, 10).tolist() == [30, 31, 32, 33]
    assert O.resident_slot_row(1, 0, 5, 1).tolist() == [5]


def test_layer_step_reads_pool_rows_for_slotted_tokens():
    """The whole unit with pool and host rows that differ: tokens whose slot
    is a pool row must be read from the pool, the cold ones from the host
    history.  The reference picks the rows by the slot row itself and runs
    torch's fp64 scaled_dot_product_attention over them."""
    n = 12
    u = synth.unit_inputs(n, seed=31, planted_blocks=[], device="cpu")
    host = synth.kv_rows(n, seed=32).numpy()
    pooled = synth.kv_rows(n, seed=33).numpy()
    slot = np.array([-1, -1, 5, 6, -1, 7, -1, -1, 8, -1, -1, 9], dtype=np.int32)
    pool = {int(s): pooled[t] for t, s in enumerate(slot) if s >= 0}
    qb = u.q.view(torch.int16).numpy().view(np.uint16)
    res = O.layer_step(u.codes.numpy(), u.scales.view(torch.int16).numpy().view(np.uint16),
                       u.q_idx.numpy(), u.w.numpy(), qb, slot, pool, host, 2048, 1 / math.sqrt(128))
    assert res["tokens"].tolist() == list(range(n))
    rows = np.where((slot >= 0)[:, None], pooled, host)
    rt = torch.from_numpy(np.ascontiguousarray(rows)).view(torch.bfloat16).reshape(n, 2, 4, 128).double()
    K = rt[:, 0].permute(1, 0, 2).repeat_interleave(4, dim=0)
    V = rt[:, 1].permute(1, 0, 2).repeat_interleave(4, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(u.q.double().reshape(16, 1, 128), K, V,
                                                           scale=1 / math.sqrt(128))
    assert np.allclose(res["out"], ref.reshape(16, 128).numpy(), rtol=0, atol=1e-12)
