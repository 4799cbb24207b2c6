"""Seeded synthetic inputs for the QSA decode step.

This module only draws random numbers and lays them out in the byte formats
the decode step consumes. It holds none of the method's arithmetic (no
scoring, no block reduction, no selection, no attention), so the CUDA path and
the fp64 CPU oracle can both consume what it makes without sharing any of the
computation.

Formats (per token, per QSA layer):

* index key: 64 FP8-e4m3 codes + one fp16 scale = 66 bytes.  The pages give
  the 66-byte figure ("Оффлоадинг KV-кэша Qwen3.8-Flash-Next в RAM через vLLM
  без потери скорости декодирования", section "Эффективность и память"); the
  split into 64 codes + a per-token absmax scale is the reading this library
  takes.
* KV row: K[4][128] bf16 followed by V[4][128] bf16 = 2048 bytes, the row
  size the same section gives for the uncompressed cache.

Distributions: keys N(0,1) quantised with a per-token absmax fp16 scale
(scale = fp16(absmax/448), codes = RNE(k/scale) clamped to +-448); index
queries N(0,1) fp32 [8][64]; head weights U(0,1) fp32 [8]; K, V and the
attention query N(0,1) bf16.

Planted blocks: a chosen set of C4 blocks is lifted above every other block
by multiplying the fp16 scale of its four tokens by PLANT_FACTOR (a power of
two, so the product is exact).  Because a token's score is linear in its
scale, the planted blocks dominate the natural score spread.  Whether the
resulting boundary gap is large enough is not assumed here: every parity test
measures it in fp64 with the oracle before it compares selections.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

INDEX_HEADS = 8
INDEX_DIM = 64
KV_HEADS = 4
HEAD_DIM = 128
Q_HEADS = 16
ROW_BYTES = 2 * KV_HEADS * HEAD_DIM * 2  # K and V, bf16
E4M3_MAX = 448.0
PLANT_FACTOR = 64.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def mix_seed(*parts: int) -> int:
    """Deterministic 63-bit seed from a tuple of small integers (splitmix64)."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x = z ^ (z >> 31)
    return x & 0x7FFF_FFFF_FFFF_FFFF


def index_keys(n: int, seed: int, device="cpu", chunk: int = 1 << 20):
    """Quantised index keys for n tokens.

    Returns (codes uint8 [n][64], scales fp16 [n]).  A token whose key is all
    zero gets scale 0 and zero codes.
    """
    codes = torch.empty(n, INDEX_DIM, dtype=torch.uint8, device=device)
    scales = torch.empty(n, dtype=torch.float16, device=device)
    g = _gen(seed, device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        k = torch.randn(e - s, INDEX_DIM, generator=g, device=device, dtype=torch.float32)
        amax = k.abs().amax(dim=1)
        sc = (amax / E4M3_MAX).to(torch.float16)
        scf = sc.float()
        safe = torch.where(scf > 0, scf, torch.ones_like(scf))
        x = (k / safe[:, None]).clamp(-E4M3_MAX, E4M3_MAX)
        x = torch.where((scf > 0)[:, None], x, torch.zeros_like(x))
        codes[s:e] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        scales[s:e] = sc
    return codes, scales


def fp8_kv_rows(rows: torch.Tensor) -> torch.Tensor:
    """FP8 rows (uint8 [m][1040]) of BF16 KV rows (uint8 [m][2048]): each of
    the 8 head vectors (K heads 0-3, V heads 0-3, 128 values) gets the index
    keys' recipe - scale = fp16(absmax/448), codes = E4M3 of clamp(x/scale,
    +-448), zero codes for a zero scale - stored as codes K[4][128],
    V[4][128], then the 8 fp16 scales."""
    m = rows.shape[0]
    x = rows.contiguous().view(torch.bfloat16).float().view(m, 8, 128)
    sc = (x.abs().amax(dim=2) / E4M3_MAX).to(torch.float16)
    scf = sc.float()
    safe = torch.where(scf > 0, scf, torch.ones_like(scf))
    q = (x / safe[:, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
    q = torch.where((scf > 0)[:, :, None], q, torch.zeros_like(q))
    out = torch.empty(m, 1040, dtype=torch.uint8, device=rows.device)
    out[:, :1024] = q.to(torch.float8_e4m3fn).view(torch.uint8).view(m, 1024)
    out[:, 1024:] = sc.contiguous().view(torch.uint8).view(m, 16)
    return out


def plant(scales: torch.Tensor, blocks, n: int, factor: float = PLANT_FACTOR):
    """Multiply the fp16 scale of every token of the given C4 blocks by factor."""
    blocks = torch.as_tensor(blocks, dtype=torch.int64, device=scales.device)
    if blocks.numel() == 0:
        return scales
    toks = (blocks[:, None] * 4 + torch.arange(4, device=scales.device)[None, :]).reshape(-1)
    toks = toks[toks < n]
    scales[toks] = (scales[toks].float() * factor).to(torch.float16)
    return scales



def unplant(scales: torch.Tensor, blocks, n: int, factor: float = PLANT_FACTOR):
    """Undo plant() on the given blocks (exact: factor is a power of two)."""
    blocks = torch.as_tensor(blocks, dtype=torch.int64, device=scales.device)
    if blocks.numel() == 0:
        return scales
    toks = (blocks[:, None] * 4 + torch.arange(4, device=scales.device)[None, :]).reshape(-1)
    toks = toks[toks < n]
    scales[toks] = (scales[toks].float() / factor).to(torch.float16)
    return scales


def drift_blocks(planted, lo: int, hi: int, frac: float, seed: int):
    """Selection drift between decode steps: of the planted blocks in
    [lo, hi), replace round(frac * count) (drawn at random) by as many
    unplanted blocks of [lo, hi).  Returns (dropped, added, new planted set)
    as sorted int64 tensors."""
    g = _gen(seed, "cpu")
    planted = torch.as_tensor(planted, dtype=torch.int64)
    inside = planted[(planted >= lo) & (planted < hi)]
    k = int(round(frac * inside.numel()))
    k = min(k, (hi - lo) - inside.numel())
    if k <= 0:
        e = torch.empty(0, dtype=torch.int64)
        return e, e, planted.sort().values
    dropped = inside[torch.randperm(inside.numel(), generator=g)[:k]].sort().values
    taken = torch.zeros(hi - lo, dtype=torch.bool)
    taken[inside - lo] = True
    free = torch.nonzero(~taken).reshape(-1) + lo
    added = free[torch.randperm(free.numel(), generator=g)[:k]].sort().values
    keep = planted[~torch.isin(planted, dropped)]
    return dropped, added, torch.cat([keep, added]).sort().values

def index_query(seed: int, device="cpu"):
    """Index query q[8][64] ~ N(0,1) fp32 and head weights w[8] ~ U(0,1) fp32."""
    g = _gen(seed, device)
    q = torch.randn(INDEX_HEADS, INDEX_DIM, generator=g, device=device, dtype=torch.float32)
    w = torch.rand(INDEX_HEADS, generator=g, device=device, dtype=torch.float32)
    return q, w


def index_query_skewed(seed: int, span_log2: float = 12.0, device="cpu"):
    """Index query with skewed magnitudes: every element is a random sign
    times 2^(-span_log2 * u), u ~ U(0,1), so the elements spread
    log-uniformly over [2^-span_log2, 1] of the largest one; head weights
    U(0,1) fp32 [8] as in index_query."""
    g = _gen(seed, device)
    u = torch.rand(INDEX_HEADS, INDEX_DIM, generator=g, device=device, dtype=torch.float64)
    sgn = torch.randint(0, 2, (INDEX_HEADS, INDEX_DIM), generator=g, device=device) * 2 - 1
    q = (sgn * torch.exp2(-span_log2 * u)).to(torch.float32)
    w = torch.rand(INDEX_HEADS, generator=g, device=device, dtype=torch.float32)
    return q, w


def attn_query(seed: int, device="cpu"):
    """Attention query [16][128] bf16 ~ N(0,1)."""
    g = _gen(seed, device)
    return torch.randn(Q_HEADS, HEAD_DIM, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def kv_rows_into(dst_u8: torch.Tensor, seed: int, gen_device="cpu", chunk_rows: int = 1 << 18):
    """Fill dst (uint8 [m][2048], any device, pinned host allowed) with KV rows.

    Each row is K[4][128] then V[4][128], bf16 N(0,1).  Rows are drawn on
    gen_device in chunks and copied into dst.
    """
    m = dst_u8.shape[0]
    g = _gen(seed, gen_device)
    for s in range(0, m, chunk_rows):
        e = min(m, s + chunk_rows)
        x = torch.randn(e - s, ROW_BYTES // 2, generator=g, device=gen_device,
                        dtype=torch.float32).to(torch.bfloat16)
        dst_u8[s:e].copy_(x.view(torch.uint8).view(e - s, ROW_BYTES), non_blocking=False)
    return dst_u8


def kv_rows(m: int, seed: int, device="cpu"):
    out = torch.empty(m, ROW_BYTES, dtype=torch.uint8, device=device)
    return kv_rows_into(out, seed, gen_device=device)


# ---------------------------------------------------------------- planting

def planted_uniform(n_blocks: int, k: int, seed: int):
    """k distinct block ids drawn uniformly from [0, n_blocks)."""
    g = _gen(seed, "cpu")
    k = min(k, n_blocks)
    return torch.randperm(n_blocks, generator=g)[:k].sort().values


def planted_hot_cold(n_blocks: int, k: int, tail_blocks: int, seed: int):
    """Half of k planted blocks inside the last tail_blocks blocks, half before."""
    g = _gen(seed, "cpu")
    k = min(k, n_blocks)
    tail_blocks = min(tail_blocks, n_blocks)
    cold = n_blocks - tail_blocks
    k_hot = min(tail_blocks, k - min(cold, k // 2))
    k_cold = k - k_hot
    hot = torch.randperm(tail_blocks, generator=g)[:k_hot] + cold
    cld = torch.randperm(cold, generator=g)[:k_cold] if k_cold > 0 else torch.empty(0, dtype=torch.int64)
    return torch.cat([cld, hot]).sort().values


def planted_zipf_sinks(n_blocks: int, k: int, seed: int, alpha: float = 1.1, n_sinks: int = 4):
    """Sink blocks 0..n_sinks-1 plus k-n_sinks blocks from a 50/50 mixture of a
    recency Zipf(alpha) law (p(d) ~ d^-alpha, d = 1 + distance from the newest
    block) and a uniform law, without replacement."""
    g = _gen(seed, "cpu")
    k = min(k, n_blocks)
    sinks = list(range(min(n_sinks, k)))
    chosen = set(sinks)
    d = torch.arange(1, n_blocks + 1, dtype=torch.float64)
    pz = d.pow(-alpha)
    pz /= pz.sum()
    while len(chosen) < k:
        need = k - len(chosen)
        nz = need // 2 + 1
        z = torch.multinomial(pz, nz, replacement=True, generator=g)
        blocks_z = (n_blocks - 1 - z).tolist()
        blocks_u = torch.randint(0, n_blocks, (need,), generator=g).tolist()
        for b in blocks_z + blocks_u:
            if len(chosen) >= k:
                break
            chosen.add(int(b))
    return torch.tensor(sorted(chosen), dtype=torch.int64)


def log_uniform_contexts(n_req: int, lo: int, hi: int, seed: int, multiple: int = 4):
    """Context lengths log-uniform in [lo, hi], rounded to a multiple."""
    g = _gen(seed, "cpu")
    u = torch.rand(n_req, generator=g, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    x = (torch.round(x / multiple) * multiple).to(torch.int64).clamp(lo, hi)
    return [int(v) for v in x.tolist()]


@dataclass
class UnitInputs:
    """Inputs of one (request, layer) decode unit on one device."""
    n: int
    codes: torch.Tensor    # uint8 [n][64]
    scales: torch.Tensor   # fp16 [n]
    q_idx: torch.Tensor    # fp32 [8][64]
    w: torch.Tensor        # fp32 [8]
    q: torch.Tensor        # bf16 [16][128]
    planted: torch.Tensor  # int64 block ids


def unit_inputs(n: int, seed: int, planted_blocks, device="cpu") -> UnitInputs:
    codes, scales = index_keys(n, mix_seed(seed, 1), device=device)
    plant(scales, planted_blocks, n)
    q_idx, w = index_query(mix_seed(seed, 2), device=device)
    q = attn_query(mix_seed(seed, 3), device=device)
    return UnitInputs(n, codes, scales, q_idx, w, q,
                      torch.as_tensor(planted_blocks, dtype=torch.int64))
