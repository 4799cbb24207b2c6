"""fp64 CPU oracle for the QSA decode step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
the CPU-baseline leg of the benchmark may import this module.  The product
path (the CUDA library and its Python binding) never calls it, and it shares
no code with that path: it decodes the byte formats itself, from their
published definitions, and computes everything in float64 with plain numpy.

What it computes, step by step (one decode unit = one request at one QSA
layer):

1. Index score per cached token t (the resident indexer over compact keys:
   "Оффлоадинг KV-кэша Qwen3.8-Flash-Next в RAM через vLLM без потери скорости
   декодирования", section "Механизм гибридного разреженного оффлоадинга"):
       S_t = sum_h w_h * relu( sum_d q_{h,d} * k_{t,d} ),   k_{t,d} = sc_t * e4m3(code_{t,d})
   with 8 index heads of 64 dims.  The dequantised key is code times scale,
   which is this library's reading of "64 FP8 values plus one fp16 scale".
2. C4 block score: the maximum of the (up to) four token scores of each
   group of four adjacent tokens ("双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测",
   the opening explanation of QSA and its C4 blocks).
3. Selection: the K = min(budget/4, #blocks) blocks that rank highest under
   the total order (score descending, block id ascending), returned in
   ascending block id.  Each layer selects on its own (same page, same part:
   the 12 sparse layers choose independently).
4. Gather through the logical-token -> physical-slot table: slot >= 0 reads
   row `slot` of the HBM pool, slot == -1 reads the token's row in the host
   store (same page, section "显存账本：热缓存卸载省下约84%": logical token
   addresses are kept apart from physical cache slots; missing blocks come
   back from pinned host memory on demand).
5. GQA decode attention over the gathered rows: query head h uses KV head
   h // 4, logits = scale * q_h . K_i, softmax over the selected tokens,
   output = sum_i p_i V_i, plus lse_h = log sum_i exp(logit_i).

Beside the step: the producer side (quantising and storing a new token's
index key and KV row, with the slot-table writes), FP8 KV rows, and the
cross-step hot cache (hot_cache_step: which selected cold tokens are copied
into a unit's hot HBM rows, and which tokens those rows held go cold).

Every function below names the passage it follows.  Pins that tie this
oracle to facts outside itself live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

INDEX_HEADS = 8
INDEX_DIM = 64
KV_HEADS = 4
HEAD_DIM = 128
Q_HEADS = 16
GQA_GROUP = Q_HEADS // KV_HEADS
ROW_BYTES = 2048
ROW_BYTES_FP8 = 1040


# ------------------------------------------------------------------ formats

def e4m3_value(code: int) -> float:
    """Value of one FP8 E4M3 code (OCP 8-bit floating point specification,
    E4M3 variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
    exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there
    is no infinity, so S.1111.110 = 448 is the largest finite value."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def decode_fp16(bits) -> np.ndarray:
    """IEEE 754 binary16 from raw bits: 1 sign, 5 exponent (bias 15), 10
    mantissa; exponent 0 = subnormal m * 2^-24; exponent 31 = inf/NaN."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = np.where(b & 0x8000, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    m = (b & 0x3FF).astype(np.float64)
    sub = m * 2.0 ** -24
    nrm = (1.0 + m / 1024.0) * np.exp2(e.astype(np.float64) - 15.0)
    special = np.where(m == 0, np.inf, np.nan)
    v = np.where(e == 0, sub, np.where(e == 31, special, nrm))
    return s * v


def decode_bf16(bits) -> np.ndarray:
    """bfloat16 from raw bits: the upper 16 bits of an IEEE binary32
    (1 sign, 8 exponent with bias 127, 7 mantissa)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = np.where(b & 0x8000, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    m = (b & 0x7F).astype(np.float64)
    sub = m * 2.0 ** (-126 - 7)
    nrm = (1.0 + m / 128.0) * np.exp2(e.astype(np.float64) - 127.0)
    special = np.where(m == 0, np.inf, np.nan)
    v = np.where(e == 0, sub, np.where(e == 255, special, nrm))
    return s * v


# ------------------------------------------------------------ 1. index score

def token_scores(codes, scale_bits, q_idx, w) -> np.ndarray:
    """S_t for every token (step 1 above; resident indexer of the offload
    digest, section "Механизм гибридного разреженного оффлоадинга").

    codes: uint8 [n][64] e4m3; scale_bits: uint16 [n] fp16 bits;
    q_idx: [8][64] float; w: [8] float.  Returns float64 [n].
    """
    k = decode_e4m3(codes) * decode_fp16(scale_bits)[:, None]          # [n][64]
    dots = k @ np.asarray(q_idx, dtype=np.float64).T                     # [n][8]
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)      # [n]


# ----------------------------------------------------------- 2. C4 blocks

def c4_block_scores(S) -> np.ndarray:
    """Block b covers tokens 4b..4b+3 (fewer in a ragged last block); its
    score is the maximum of its tokens' scores (C4 grouping, RTX4090 port
    page, opening explanation of QSA)."""
    S = np.asarray(S, dtype=np.float64)
    n = S.shape[0]
    nb = (n + 3) // 4
    out = np.empty(nb, dtype=np.float64)
    for b in range(nb):
        out[b] = S[4 * b:min(n, 4 * b + 4)].max()
    return out


# -------------------------------------------------------------- 3. top-k

def select_blocks(blk, budget_tokens: int) -> np.ndarray:
    """The K = min(budget_tokens // 4, #blocks) highest-ranking blocks under
    (score descending, block id ascending), sorted by block id (per-layer
    independent selection within indexer_budget: offload digest lead and
    section "Механизм гибридного разреженного оффлоадинга"; RTX4090 port page,
    opening explanation of QSA)."""
    blk = np.asarray(blk, dtype=np.float64)
    nb = blk.shape[0]
    k = min(budget_tokens // 4, nb)
    ids = np.arange(nb)
    order = np.lexsort((ids, -blk))      # primary: -score, secondary: id
    return np.sort(order[:k]).astype(np.int64)


def selected_tokens(sel_blocks, n: int) -> np.ndarray:
    """Token positions covered by the selected blocks, ascending, without the
    positions past the end of the context."""
    toks = [t for b in np.asarray(sel_blocks, dtype=np.int64)
            for t in range(4 * int(b), min(n, 4 * int(b) + 4))]
    return np.asarray(toks, dtype=np.int64)


# ------------------------------------------------ 4. slot-table gather

def ring_slot_row(ctx_len: int, layer: int, base_row: int, ring_tokens: int) -> np.ndarray:
    """Slot-table row of one layer of a host-offloaded request: the newest
    ring_tokens tokens live in the request's tail ring (token t in ring row
    t mod ring_tokens of that layer's ring), every older token is cold
    (-1, served from pinned host memory).  RTX4090 port page, section
    "显存账本：热缓存卸载省下约84%" (tail ring buffer; full history in pinned
    host memory; logical addresses separate from physical slots)."""
    t = np.arange(ctx_len, dtype=np.int64)
    hot = t >= ctx_len - ring_tokens
    slots = base_row + layer * ring_tokens + (t % ring_tokens)
    return np.where(hot, slots, -1).astype(np.int32)


def resident_slot_row(ctx_len: int, layer: int, base_row: int,
                      layer_rows: int | None = None) -> np.ndarray:
    """Slot-table row of one layer of a fully HBM-resident request: token t
    of layer l sits in row base_row + l * layer_rows + t, where layer_rows is
    the region's rows per layer (the request's capacity; ctx_len when it was
    leased without room to grow)."""
    stride = ctx_len if layer_rows is None else layer_rows
    return (base_row + layer * stride + np.arange(ctx_len, dtype=np.int64)).astype(np.int32)


def gather_rows(tokens, slot_row, hbm_pool_rows, host_rows, row_bytes: int = ROW_BYTES) -> np.ndarray:
    """Bytes of the rows of the given logical tokens: pool row slot_row[t]
    when it is >= 0, else host row t (step 4 above).  Returns uint8
    [m][row_bytes].  hbm_pool_rows / host_rows: anything indexable by row
    giving row_bytes bytes (2048 for bf16 rows, 1040 for FP8 rows)."""
    out = np.empty((len(tokens), row_bytes), dtype=np.uint8)
    for i, t in enumerate(tokens):
        s = int(slot_row[int(t)])
        out[i] = hbm_pool_rows[s] if s >= 0 else host_rows[int(t)]
    return out



def hot_cache_step(tokens, slot_row, owner, cursor: int, hot_base: int):
    """One decode step of a unit's cross-step hot cache.  RTX4090 port page,
    section "显存账本：热缓存卸载省下约84%": the full history stays in pinned
    host memory, missing blocks are moved back to the GPU on demand, and the
    GPU keeps a hot cache whose rows are found through the slot table.  This
    library's reading: the unit owns H = len(owner) pool rows hot_base ..
    hot_base + H - 1; owner[v] is the token row v holds (-1: none) and
    `cursor` the next row to hand out.  For the selected tokens (ascending):
      - a token whose slot is one of the unit's hot rows is a hit; its row is
        in use by this step;
      - a token whose slot is -1 is a miss; misses take rows in ascending
        token order;
      - the rows handed out are the first rows not in use by this step in the
        circular order cursor, cursor + 1, ... (mod H); when there are fewer
        such rows than misses, the remaining misses stay cold;
      - a row's previous owner e becomes cold (slot -1) if its slot still
        names that row (a slot remapped elsewhere is left alone);
      - the miss takes the row (owner, slot) and its host row is copied in;
      - the cursor moves one past the last row handed out.
    Tokens whose slot is any other pool row (tail ring, staging) are left
    alone.  Returns (new slot row, new owner, new cursor, fills) with fills
    the (token, pool row) pairs whose host rows are copied."""
    slot = np.array(slot_row, dtype=np.int32, copy=True)
    own = np.array(owner, dtype=np.int32, copy=True)
    H = len(own)
    in_use = set()
    misses = []
    for t in sorted(int(x) for x in tokens):
        s_ = int(slot[t])
        if hot_base <= s_ < hot_base + H:
            in_use.add(s_ - hot_base)
        elif s_ == -1:
            misses.append(t)
    rows = []
    k = 0
    while len(rows) < len(misses) and k < H:
        v = (cursor + k) % H
        if v not in in_use:
            rows.append(v)
        k += 1
    fills = []
    for t, v in zip(misses, rows):
        e = int(own[v])
        if e >= 0 and int(slot[e]) == hot_base + v:
            slot[e] = -1
        own[v] = t
        slot[t] = hot_base + v
        fills.append((t, hot_base + v))
    if rows:
        cursor = (rows[-1] + 1) % H
    return slot, own, int(cursor), fills


# ----------------------------------------------------------- 5. attention

def split_kv(rows_u8) -> tuple[np.ndarray, np.ndarray]:
    """A 2048-byte row holds K[4][128] bf16 then V[4][128] bf16."""
    r = np.ascontiguousarray(rows_u8, dtype=np.uint8).view(np.uint16).reshape(-1, 2, KV_HEADS, HEAD_DIM)
    return decode_bf16(r[:, 0]), decode_bf16(r[:, 1])          # [m][4][128] each


def split_kv_fp8(rows_u8) -> tuple[np.ndarray, np.ndarray]:
    """A 1040-byte FP8 row holds K codes [4][128] E4M3, V codes [4][128]
    E4M3, then fp16 scales for K heads 0-3 and V heads 0-3; an element's
    value is its head's scale times e4m3(code).  This is the library's
    reading of an FP8 KV cache: the RTX 5090 page runs one (FP8 KV), and the
    RTX4090 port's per-card memory figure fits about 1 KiB per token and
    layer.  The per-head absmax scale is the same reading as the index
    key's."""
    r = np.ascontiguousarray(rows_u8, dtype=np.uint8).reshape(-1, ROW_BYTES_FP8)
    kc = r[:, :512].reshape(-1, KV_HEADS, HEAD_DIM)
    vc = r[:, 512:1024].reshape(-1, KV_HEADS, HEAD_DIM)
    sc = np.ascontiguousarray(r[:, 1024:1040]).view(np.uint16).reshape(-1, 2, KV_HEADS)
    ks, vs = decode_fp16(sc[:, 0]), decode_fp16(sc[:, 1])      # [m][4]
    return decode_e4m3(kc) * ks[:, :, None], decode_e4m3(vc) * vs[:, :, None]


def decode_attention(q_bits, rows_u8, softmax_scale: float, kv_format: str = "bf16"):
    """GQA decode attention over the gathered rows (step 5 above; sparse
    attention over the selected rows only, offload digest section
    "Механизм гибридного разреженного оффлоадинга").  kv_format "bf16":
    2048-byte rows (split_kv); "fp8": 1040-byte rows (split_kv_fp8).

    q_bits: uint16 [16][128] bf16 bits.  Returns (out float64 [16][128],
    lse float64 [16]); with no rows, out = 0 and lse = -inf.
    """
    q = decode_bf16(q_bits).reshape(Q_HEADS, HEAD_DIM)
    out = np.zeros((Q_HEADS, HEAD_DIM))
    lse = np.full(Q_HEADS, -np.inf)
    if len(rows_u8) == 0:
        return out, lse
    K, V = split_kv(rows_u8) if kv_format == "bf16" else split_kv_fp8(rows_u8)
    for h in range(Q_HEADS):
        g = h // GQA_GROUP
        logits = softmax_scale * (K[:, g, :] @ q[h])               # [m]
        m = logits.max()
        p = np.exp(logits - m)
        l = p.sum()
        out[h] = (p @ V[:, g, :]) / l
        lse[h] = m + np.log(l)
    return out, lse


# ------------------------------------------------------- whole layer-step

def layer_step(codes, scale_bits, q_idx, w, q_bits, slot_row, hbm_pool_rows,
               host_rows, budget_tokens: int, softmax_scale: float):
    """One decode unit end to end: steps 1-5 in the order the pages give
    them (score every cached token, pick at most indexer_budget tokens by C4
    blocks, bring only those rows, attend over them)."""
    n = np.asarray(codes).shape[0]
    S = token_scores(codes, scale_bits, q_idx, w)
    blk = c4_block_scores(S)
    sel = select_blocks(blk, budget_tokens)
    toks = selected_tokens(sel, n)
    rows = gather_rows(toks, slot_row, hbm_pool_rows, host_rows)
    out, lse = decode_attention(q_bits, rows, softmax_scale)
    return dict(scores=S, blk=blk, sel=sel, tokens=toks, out=out, lse=lse)


def boundary_gap(blk, budget_tokens: int) -> float:
    """Score gap between the last selected block and the best unselected one
    (inf when every block is selected)."""
    blk = np.asarray(blk, dtype=np.float64)
    k = min(budget_tokens // 4, blk.shape[0])
    if k >= blk.shape[0]:
        return float("inf")
    s = np.sort(blk)[::-1]
    return float(s[k - 1] - s[k])


# ------------------------------------------------ 6. producer side: append

# The 127 non-negative finite E4M3 values in code order (codes 0x00..0x7E):
# the magnitude encoding is monotonic, so code order is value order.
E4M3_POSITIVE = np.array([e4m3_value(c) for c in range(0x7F)], dtype=np.float64)


def encode_e4m3(x) -> np.ndarray:
    """FP8 E4M3 code of each value (OCP 8-bit floating point specification,
    E4M3 variant, as e4m3_value above): round to nearest, a value halfway
    between two neighbours goes to the one with the even code, magnitudes
    above the largest finite value 448 saturate to 448 (E4M3 has no
    infinity).  The sign bit follows the sign of the input, so -0.0 and
    negative values that round to zero give 0x80."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(E4M3_POSITIVE, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = E4M3_POSITIVE[hi] - a
    d_lo = a - E4M3_POSITIVE[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def quantize_vector(x) -> tuple[np.ndarray, int]:
    """Codes and scale bits of one vector under the producer's rule (see
    quantize_index_key); shared by index keys and FP8 KV rows."""
    return quantize_index_key(x)


def quantize_index_key(k) -> tuple[np.ndarray, int]:
    """Index key of a new token as the producer stores it: 64 FP8-e4m3 codes
    and one fp16 scale (the 66-byte key of the offload digest, section
    "Эффективность и память"; split into codes + per-token absmax scale as
    this library reads it).  The rounding decisions are taken in fp32, the
    precision the key arrives in:
      scale = binary16 round-to-nearest-even of (absmax / 448), the division
              in fp32; a quotient above the largest finite binary16 (65504)
              saturates to 65504;
      code_d = encode_e4m3(clamp(k_d / scale, -448, 448)), the division in fp32.
    A key whose scale is 0 (all zeros, or absmax / 448 below the smallest
    binary16) keeps scale 0 and 64 zero codes.  Returns (codes uint8 [64],
    scale bits uint16)."""
    k = np.asarray(k, dtype=np.float32).reshape(-1)
    amax = np.float32(np.max(np.abs(k)))
    q = np.float32(amax / np.float32(448.0))
    q = np.minimum(q, np.float32(65504.0))
    s16 = np.float16(q)
    if s16 == 0:
        return np.zeros(k.size, dtype=np.uint8), 0
    x = (k / np.float32(s16)).astype(np.float32)
    x = np.clip(x, np.float32(-448.0), np.float32(448.0))
    return encode_e4m3(x), int(np.array(s16).view(np.uint16))


def append_slot_writes(t: int, placement: str, base_row: int, layer: int, layer_rows: int,
                       ring_tokens: int) -> list:
    """Slot-table writes, as (token, slot) pairs, when token t - the newest
    one of its request - is stored at one layer.  RTX4090 port page, section
    "显存账本：热缓存卸载省下约84%" (full history in pinned host memory, a tail
    ring buffer of the newest tokens in HBM, logical tokens kept apart from
    physical slots):
      "hbm":  the token's own row base_row + layer*layer_rows + t;
      "host": cold (-1), its row lives in the host history only;
      "ring": ring row base_row + layer*ring_tokens + (t mod ring_tokens),
              and the token that held that ring row before, t - ring_tokens,
              becomes cold (its row stays in the host history)."""
    if placement == "hbm":
        return [(t, base_row + layer * layer_rows + t)]
    if placement == "host":
        return [(t, -1)]
    if placement == "ring":
        w = [(t, base_row + layer * ring_tokens + t % ring_tokens)]
        if t >= ring_tokens:
            w.append((t - ring_tokens, -1))
        return w
    raise ValueError(placement)


def quantize_kv_row_fp8(row_u8) -> np.ndarray:
    """FP8 row (1040 bytes, layout of split_kv_fp8) of a bf16 KV row (2048
    bytes, layout of split_kv): each of the 8 vectors K[h], V[h] (128 values,
    exact in fp32) is quantised under the index key's rule - fp16 scale =
    round-to-nearest-even of absmax/448 in fp32, E4M3 codes of clamp(x/scale,
    +-448) - and stored as codes K[4][128], V[4][128], scales K[4], V[4]."""
    bits = np.ascontiguousarray(row_u8, dtype=np.uint8).view(np.uint16).reshape(2, KV_HEADS, HEAD_DIM)
    vals = decode_bf16(bits).astype(np.float32)
    out = np.zeros(ROW_BYTES_FP8, dtype=np.uint8)
    scales = np.zeros(2 * KV_HEADS, dtype=np.uint16)
    for kv in range(2):
        for h in range(KV_HEADS):
            codes, sbits = quantize_vector(vals[kv, h])
            off = kv * 512 + h * HEAD_DIM
            out[off:off + HEAD_DIM] = codes
            scales[kv * KV_HEADS + h] = sbits
    out[1024:1040] = scales.view(np.uint8)
    return out
