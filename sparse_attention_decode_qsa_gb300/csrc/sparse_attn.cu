// Step 4 of the QSA decode step: GQA decode attention over the selected
// rows only ("Оффлоадинг KV-кэша Qwen3.8-Flash-Next в RAM через vLLM без
// потери скорости декодирования", section "Механизм гибридного разреженного
// оффлоадинга": attention reads only the <= indexer_budget selected rows).
//
// Split-K flash-decode.  A split is 4 selected C4 blocks, i.e. 16 token
// rows.  Rows are read through the slot table (pool rows from HBM, cold rows
// zero-copy from mapped pinned host memory) or from a dense gathered buffer.
//
// Work layout: unit u gets cpu_u CTAs (cta_start holds their prefix sums);
// CTA (unit u, slot r) takes the splits r, r + cpu_u, r + 2*cpu_u, ... of
// unit u and visits them alternately from the front and the back of that
// list.  Selected blocks are in ascending id order, so for a request with an
// HBM tail ring the early splits are cold (host) and the late ones hot (HBM):
// the alternation overlaps host transfers with compute.  The units that read
// host memory share kMaxCtasHost CTAs: that many SMs saturate the host link,
// and the others stay free for HBM-bound work of other requests on other
// streams.  Units that read only HBM share the rest of the SMs.
//
// Inside a CTA the 8 warps work independently: warp w serves KV head
// g = w % 4 (its 4 query heads) for tokens 8*(w/4) .. 8*(w/4)+7 of every
// split.  A warp copies only its KV head's 512 bytes of each of its 8 rows
// (K[g] then V[g]) with cp.async into its own double buffer (64 KiB per CTA,
// small enough to share an SM with the index-score CTAs), so no CTA-wide
// barrier is needed while streaming; it keeps a running online-softmax state
// (max, sum, acc) for its 4 heads over all its tokens.  At the end the two
// token halves of each KV head are merged in shared memory and the CTA writes
// one partial; a small second kernel merges the cpu partials of each
// (unit, head) with the log-sum-exp rule.  (Merging in the split kernel's
// last CTA per unit was measured: the extra epilogue code halved the
// streaming loop's host-read rate, even on launches that did not run it.)
//
// Per warp and split: logits with lane l holding dims 4l..4l+3 of the 4 query
// heads, reduced across the warp with a transposing butterfly (6 shuffles
// for 4 values); after it the lanes 8j..8j+7 hold head j, lane 8j+k keeping
// token k.  Softmax statistics are reduced over those 8 lanes; P.V
// broadcasts each token's 4 probabilities with shuffles and accumulates dims
// 4l..4l+3.  Plain FMAs throughout: 4 query heads per KV head make this a
// 4-row contraction, not a tensor-core shape.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

#ifndef QSA_PDL_TRIGGER_MERGE
#define QSA_PDL_TRIGGER_MERGE 1
#endif

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBlocksPerSplit = 4;                    // selected C4 blocks per split
constexpr int kWarpTokens = 8;                        // tokens per warp and split
constexpr int kSliceBytes = 2 * kHeadDim * 2;         // K[g] + V[g] of one token: 512
constexpr int kWarpBufBytes = kWarpTokens * kSliceBytes;  // 4 KiB
#ifndef QSA_ATTN_STAGES
#define QSA_ATTN_STAGES 2
#endif
constexpr int kAStages = QSA_ATTN_STAGES;                 // splits in flight per warp
constexpr int kSmemBytes = kWarps * kAStages * kWarpBufBytes;  // 64 KiB at 2 stages
#ifndef QSA_ATTN_HOST_CTAS
#define QSA_ATTN_HOST_CTAS 32
#endif
constexpr int kMaxCtasHost = QSA_ATTN_HOST_CTAS;
// CTAs per SM that units reading only HBM share
#ifndef QSA_ATTN_HBM_CTAS_PER_SM
#define QSA_ATTN_HBM_CTAS_PER_SM 1
#endif
constexpr int kHbmCtasPerSm = QSA_ATTN_HBM_CTAS_PER_SM;
// Register budget per thread: at 80 one CTA (20 K registers) fits on an SM
// beside two index-score CTAs.
#ifndef QSA_ATTN_MAXREG
#define QSA_ATTN_MAXREG 80
#endif
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  BatchDesc b;
  const uint16_t* q;        // [units][16][128] bf16 bits
  const int32_t* sel;       // [units][k_max]
  const int32_t* n_sel;
  int32_t k_max;
  int32_t budget_tokens;
  int32_t cta_start[kMaxUnits + 1];  // prefix sums of the CTAs (partials) per unit
  const uint8_t* gathered;  // [units][budget_tokens][2048] or nullptr
  float scale_log2;         // softmax_scale * log2(e)
  float* out;               // [units][16][128]
  float* lse;               // [units][16] or nullptr
};

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ float* partial_ptr(const BatchDesc& b, int u, int slot) {
  const int64_t rl = (int64_t)b.u[u].req * b.n_layers + b.u[u].layer;
  return b.partials + (rl * b.splits_max + slot) * kPartFloats;
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint32_t src_bytes) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Unit u of CTA `cta`, its slot r among the unit's CTAs and their number cpu.
__device__ __forceinline__ void cta_unit(const AttnParams& p, int cta, int& u, int& r, int& cpu) {
  int lo = 0, hi = p.b.n_units - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cta_start[mid] <= cta) lo = mid; else hi = mid - 1;
  }
  u = lo;
  r = cta - p.cta_start[lo];
  cpu = p.cta_start[lo + 1] - p.cta_start[lo];
}

// The k-th split this CTA visits (0 <= k < count): alternately from the front
// and the back of its list r, r + cpu, ...
__device__ __forceinline__ int visit_split(int k, int count, int r, int cpu) {
  const int idx = (k & 1) ? count - 1 - (k >> 1) : (k >> 1);
  return r + idx * cpu;
}

// Row code of token `tok` (0..15) of a split: >= 0 a pool row (with gathered
// rows, a row of that buffer), -1 no row (past the selection or the
// context, or invalid), <= -2 the host row of token -code - 2 (a cold token,
// or a miss planned by qsa_hot_cache_plan, whose hot row goes to *dst_row).
// Reads the selection, the pending map and the slot table.
__device__ __forceinline__ int32_t resolve_row(const AttnParams& p, int u, int split, int tok, int nsel,
                                               const int32_t* pend, int32_t* dst_row) {
  *dst_row = -1;
  const int j = split * kBlocksPerSplit + tok / 4;        // selected-block index
  if (j >= nsel) return -1;
  const int64_t n = p.b.u[u].n;
  const int64_t b = p.sel[(int64_t)u * p.k_max + j];
  const int64_t t = 4 * b + (tok & 3);
  if (b < 0 || 4 * b >= n) {
    if ((tok & 3) == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernAttn, b);
    return -1;
  }
  if (t >= n) return -1;
  const int jpos = 4 * j + (tok & 3);
  if (p.gathered) return (int32_t)((int64_t)u * p.budget_tokens + jpos);
  if (pend) {
    const int32_t row = pend[jpos];
    if (row >= 0 && (int64_t)row < p.b.pool_rows && p.b.u[u].host_rows) {
      *dst_row = row;
      return (int32_t)(-2 - t);
    }
  }
  const int32_t slot = p.b.slot_table[p.b.unit_row(u) + t];
  if (slot >= 0 && (int64_t)slot < p.b.pool_rows) return slot;
  if (slot == -1 && p.b.u[u].host_rows) return (int32_t)(-2 - t);
  report_error(p.b.err, QSA_ERR_BAD_SLOT, kKernAttn, ((int64_t)u << 40) | (t & 0xFFFFFFFFFFll));
  return -1;
}

__device__ __forceinline__ const uint8_t* row_ptr(const AttnParams& p, int u, int32_t code) {
  if (code == -1) return nullptr;
  if (code >= 0) return (p.gathered ? p.gathered : p.b.pool) + (int64_t)code * p.b.row_bytes;
  return p.b.u[u].host_rows + (-2 - (int64_t)code) * p.b.row_bytes;
}

// The pending map of unit u when qsa_hot_cache_plan left copies to this
// launch, else nullptr.
__device__ __forceinline__ const int32_t* pending_map(const AttnParams& p, int u) {
  if (p.gathered || !p.b.hot_pend || p.b.u[u].hot_base < 0) return nullptr;
  const int64_t st = p.b.unit_state(u);
  return p.b.hot_pend_on[st] ? p.b.hot_pend + st * p.b.hot_fill_stride : nullptr;
}

// Row sources resolved up front: a CTA's first kPreSplits splits (16 rows
// each, in visit order) are resolved by all its threads at once, so that
// the streaming loop issues each split's row copies without first waiting
// for the selection and the slot table (two dependent global loads that
// otherwise sat in front of every split).  Later splits, if any, are
// resolved when they are issued.
#ifndef QSA_ATTN_PRESPLITS
#define QSA_ATTN_PRESPLITS 32
#endif
constexpr int kPreSplits = QSA_ATTN_PRESPLITS;
constexpr int kPreRows = (kPreSplits > 0 ? kPreSplits : 1) * kBlocksPerSplit * 4;   // 512

__device__ __forceinline__ void preload_rows(const AttnParams& p, int u, int r, int cpu, int count,
                                             int nsel, const int32_t* pend, int32_t* code,
                                             int32_t* dst) {
  const int npre = (count < kPreSplits ? count : kPreSplits) * kBlocksPerSplit * 4;
  for (int idx = threadIdx.x; idx < npre; idx += kThreads) {
    const int k = idx >> 4, tok = idx & 15;
    int32_t d;
    code[idx] = resolve_row(p, u, visit_split(k, count, r, cpu), tok, nsel, pend, &d);
    dst[idx] = d;
  }
  __syncthreads();
}

// Lane l < 8 of the warp: the source (and, for a planned miss, the hot row)
// of token half*8 + l of the k-th split the CTA visits.
__device__ __forceinline__ const uint8_t* lane_source(const AttnParams& p, int u, int k, int split,
                                                      int nsel, int half, const int32_t* pend,
                                                      const int32_t* pcode, const int32_t* pdst,
                                                      uint8_t** dst) {
  const int tok = half * kWarpTokens + (threadIdx.x & 31);
  int32_t code, drow;
  if (k < kPreSplits) {
    code = pcode[k * 16 + tok];
    drow = pdst[k * 16 + tok];
  } else {
    code = resolve_row(p, u, split, tok, nsel, pend, &drow);
  }
  *dst = drow >= 0 ? p.b.pool + (int64_t)drow * p.b.row_bytes : nullptr;
  return row_ptr(p, u, code);
}

// Copy this warp's 8 token slices (K[g], V[g]) of the k-th split it visits
// into buf.  Lane l resolves token l (l < 8); every lane then copies 16
// bytes of each slice.  Returns a bitmask of the tokens that exist.
__device__ __forceinline__ uint32_t issue_warp(const AttnParams& p, int u, int k, int split, int nsel,
                                               int g, int half, uint8_t* buf, const int32_t* pend,
                                               const int32_t* pcode, const int32_t* pdst,
                                               uint8_t** dsts) {
  const int lane = threadIdx.x & 31;
  const uint8_t* src = nullptr;
  if (lane < kWarpTokens) {
    uint8_t* dst;
    src = lane_source(p, u, k, split, nsel, half, pend, pcode, pdst, &dst);
    dsts[lane] = dst;
  }
  const uint32_t valid = __ballot_sync(0xFFFFFFFFu, src != nullptr) & ((1u << kWarpTokens) - 1u);
  // lanes 0..15 copy K[g] (chunks of 16 B), lanes 16..31 copy V[g]
  const int off = (lane < 16) ? g * kHeadDim * 2 + lane * 16
                              : kKvHeads * kHeadDim * 2 + g * kHeadDim * 2 + (lane - 16) * 16;
#pragma unroll
  for (int i = 0; i < kWarpTokens; ++i) {
    const uint8_t* s = reinterpret_cast<const uint8_t*>(
        __shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(src), i));
    cp_async16(buf + i * kSliceBytes + lane * 16, s ? s + off : p.b.pool, s ? 16u : 0u);
  }
  return valid;
}

// Copy this warp's slices of the stage's planned misses (K[g], V[g]: 16
// bytes per lane and token) from shared memory into their hot rows.
__device__ __forceinline__ void write_back(uint8_t* const* dsts, const uint8_t* R, int g, int lane) {
  const int off = (lane < 16) ? g * kHeadDim * 2 + lane * 16
                              : kKvHeads * kHeadDim * 2 + g * kHeadDim * 2 + (lane - 16) * 16;
#pragma unroll
  for (int i = 0; i < kWarpTokens; ++i) {
    uint8_t* d = dsts[i];
    if (d) *reinterpret_cast<uint4*>(d + off) = *reinterpret_cast<const uint4*>(R + i * kSliceBytes + lane * 16);
  }
}

// End of a split CTA: merge the two token halves of each KV head through
// shared memory, then write the CTA's partial (m, l, acc) for the merge.
__device__ __forceinline__ void finish_split(const AttnParams& p, int u, int r, int g, int half,
                                             int lane, int hj, float m_run, float l_run,
                                             float (&acc)[kGroup][4], float (&xm)[kKvHeads][kGroup],
                                             float (&xl)[kKvHeads][kGroup],
                                             float (&xacc)[kKvHeads][kGroup][kHeadDim]) {
  if (half == 1) {
    if ((lane & 7) == 0) { xm[g][hj] = m_run; xl[g][hj] = l_run; }
#pragma unroll
    for (int j = 0; j < kGroup; ++j)
      *reinterpret_cast<float4*>(&xacc[g][j][4 * lane]) = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
  }
  __syncthreads();
  if (half == 0) {
    const float mo = xm[g][hj], lo = xl[g][hj];
    const float mn = fmaxf(m_run, mo);
    const float sa = (mn == -INFINITY) ? 0.f : exp2f(m_run - mn);
    const float sb = (mn == -INFINITY) ? 0.f : exp2f(mo - mn);
    const float L = fmaf(l_run, sa, lo * sb);
    float* part = partial_ptr(p.b, u, r);
    if ((lane & 7) == 0) {
      part[g * kGroup + hj] = mn;
      part[kQHeads + g * kGroup + hj] = L;
    }
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const float aj = __shfl_sync(0xFFFFFFFFu, sa, 8 * j);
      const float bj = __shfl_sync(0xFFFFFFFFu, sb, 8 * j);
      const float4 o = *reinterpret_cast<const float4*>(&xacc[g][j][4 * lane]);
      *reinterpret_cast<float4*>(part + 2 * kQHeads + (g * kGroup + j) * kHeadDim + 4 * lane) =
          make_float4(fmaf(acc[j][0], aj, o.x * bj), fmaf(acc[j][1], aj, o.y * bj),
                      fmaf(acc[j][2], aj, o.z * bj), fmaf(acc[j][3], aj, o.w * bj));
    }
  }
}

__global__ void __maxnreg__(QSA_ATTN_MAXREG) attn_split_kernel(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];  // [warp][stage][8][512]
  __shared__ float xm[kKvHeads][kGroup], xl[kKvHeads][kGroup];
  __shared__ uint32_t vmask[kWarps][kAStages];     // tokens present in each stage
  __shared__ uint8_t* pdst[kWarps][kAStages][kWarpTokens];   // hot rows of planned misses
  __shared__ int32_t pre_code[kPreRows], pre_dst[kPreRows];     // resolved row sources
  __shared__ __align__(16) float xacc[kKvHeads][kGroup][kHeadDim];

  int u, r, cpu;
  cta_unit(p, blockIdx.x, u, r, cpu);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = warp & 3, half = warp >> 2;
  uint8_t* wbuf = smem + warp * kAStages * kWarpBufBytes;
  grid_dependency_wait();   // the selection is read from here on
  int nsel = p.n_sel[u];
  if (nsel < 0 || nsel > p.k_max) {
    if (r == 0 && threadIdx.x == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernAttn, nsel);
    nsel = 0;
  }
  const int splits = (nsel + kBlocksPerSplit - 1) / kBlocksPerSplit;
  const int count = r < splits ? (splits - 1 - r) / cpu + 1 : 0;

  // query dims 4l..4l+3 of the 4 heads of KV head g, pre-scaled to base 2
  float qr[kGroup][4];
  {
    const uint16_t* qu = p.q + (int64_t)u * kQHeads * kHeadDim;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const uint2 w2 = *reinterpret_cast<const uint2*>(qu + (g * kGroup + j) * kHeadDim + 4 * lane);
      qr[j][0] = bf16_lo(w2.x) * p.scale_log2;
      qr[j][1] = bf16_hi(w2.x) * p.scale_log2;
      qr[j][2] = bf16_lo(w2.y) * p.scale_log2;
      qr[j][3] = bf16_hi(w2.y) * p.scale_log2;
    }
  }
  const int hj = (lane >> 3) & 3;      // head whose statistics this lane holds
  float m_run = -INFINITY, l_run = 0.f;  // statistics of head hj (same in lanes 8hj..8hj+7)
  float acc[kGroup][4];                // dims 4l..4l+3 of the 4 heads
#pragma unroll
  for (int j = 0; j < kGroup; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  // splits k + 1 .. k + kAStages - 1 are in flight while split k is computed
  const int32_t* pend = pending_map(p, u);
  preload_rows(p, u, r, cpu, count, nsel, pend, pre_code, pre_dst);
#pragma unroll
  for (int k = 0; k < kAStages - 1; ++k) {
    if (k < count) {
      const uint32_t v = issue_warp(p, u, k, visit_split(k, count, r, cpu), nsel, g, half,
                                    wbuf + k * kWarpBufBytes, pend, pre_code, pre_dst, pdst[warp][k]);
      if (lane == 0) vmask[warp][k] = v;
    }
    cp_async_commit();
  }
  for (int k = 0; k < count; ++k) {
    const int kn = k + kAStages - 1;
    if (kn < count) {   // its buffer was last read in iteration k - 1
      const uint32_t v = issue_warp(p, u, kn, visit_split(kn, count, r, cpu), nsel, g, half,
                                    wbuf + (kn % kAStages) * kWarpBufBytes, pend, pre_code, pre_dst,
                                    pdst[warp][kn % kAStages]);
      if (lane == 0) vmask[warp][kn % kAStages] = v;
    }
    cp_async_commit();
    cp_async_wait<kAStages - 1>();
    __syncwarp();
    const uint32_t valid_cur = vmask[warp][k % kAStages];
    const uint8_t* R = wbuf + (k % kAStages) * kWarpBufBytes;
    if (pend) write_back(pdst[warp][k % kAStages], R, g, lane);

    // logits: lane 8j+kk ends with token kk of head j
    float x0 = -INFINITY;
#pragma unroll
    for (int i = 0; i < kWarpTokens; ++i) {
      const uint2 kk = *reinterpret_cast<const uint2*>(R + i * kSliceBytes + lane * 8);
      const float k0 = bf16_lo(kk.x), k1 = bf16_hi(kk.x), k2 = bf16_lo(kk.y), k3 = bf16_hi(kk.y);
      float d[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j)
        d[j] = fmaf(qr[j][3], k3, fmaf(qr[j][2], k2, fmaf(qr[j][1], k1, qr[j][0] * k0)));
      const bool up16 = lane & 16;
      const float a0 = up16 ? d[0] : d[2], a1 = up16 ? d[1] : d[3];
      const float r0 = __shfl_xor_sync(0xFFFFFFFFu, a0, 16);
      const float r1 = __shfl_xor_sync(0xFFFFFFFFu, a1, 16);
      const float v0 = (up16 ? d[2] : d[0]) + r0;
      const float v1 = (up16 ? d[3] : d[1]) + r1;
      const bool up8 = lane & 8;
      const float a = up8 ? v0 : v1;
      float v = (up8 ? v1 : v0) + __shfl_xor_sync(0xFFFFFFFFu, a, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
      if ((lane & 7) == i) x0 = ((valid_cur >> i) & 1u) ? v : -INFINITY;
    }

    // online softmax of head hj over its 8 tokens of this split
    float ms = x0;
    ms = fmaxf(ms, __shfl_xor_sync(0xFFFFFFFFu, ms, 1));
    ms = fmaxf(ms, __shfl_xor_sync(0xFFFFFFFFu, ms, 2));
    ms = fmaxf(ms, __shfl_xor_sync(0xFFFFFFFFu, ms, 4));
    const float m_new = fmaxf(m_run, ms);
    const float so = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);  // old-state scale
    const float p0 = (x0 == -INFINITY) ? 0.f : exp2f(x0 - m_new);
    float ps = p0;
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 1);
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 2);
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 4);
    l_run = fmaf(l_run, so, ps);
    m_run = m_new;

    // P.V: rescale, then add this split's tokens
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const float sj = __shfl_sync(0xFFFFFFFFu, so, 8 * j);
      acc[j][0] *= sj; acc[j][1] *= sj; acc[j][2] *= sj; acc[j][3] *= sj;
    }
#pragma unroll
    for (int i = 0; i < kWarpTokens; ++i) {
      const uint2 vv = *reinterpret_cast<const uint2*>(R + i * kSliceBytes + kHeadDim * 2 + lane * 8);
      const float v0 = bf16_lo(vv.x), v1 = bf16_hi(vv.x), v2 = bf16_lo(vv.y), v3 = bf16_hi(vv.y);
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const float pj = __shfl_sync(0xFFFFFFFFu, p0, 8 * j + i);
        acc[j][0] = fmaf(pj, v0, acc[j][0]);
        acc[j][1] = fmaf(pj, v1, acc[j][1]);
        acc[j][2] = fmaf(pj, v2, acc[j][2]);
        acc[j][3] = fmaf(pj, v3, acc[j][3]);
      }
    }
    __syncwarp();   // this buffer is refilled in the next iteration
  }
  asm volatile("cp.async.wait_all;" ::: "memory");

  finish_split(p, u, r, g, half, lane, hj, m_run, l_run, acc, xm, xl, xacc);
  trigger_dependents();
}

// ---------------------------------------------------------------------------
// FP8 rows (QSA_ROW_BYTES_FP8: E4M3 codes of K [4][128] and V [4][128], then
// fp16 scales K[4], V[4]).  Same work layout as the BF16 kernel, except
// that the four warps of a token half (one per KV head) share their rows:
// per split they copy the half's 8 rows whole (8 x 1040 bytes, 16-byte
// pieces; thread t of the half takes pieces t, t + 128, ...) into a stage
// buffer, meet at a named barrier, and each warp then reads its head's
// codes and scales from the staged rows.  A warp instruction so covers 512
// contiguous bytes of a row, as in the BF16 kernel; fetching each head's
// 128-byte code pieces and the 16 scale bytes separately (four times, once
// per head) gave 2.5 times the requests per byte and 21 % more host-memory
// sectors than the rows hold.  A token's K scale multiplies its logit after
// the dot product, its V scale its probability in P.V.
constexpr int kChunksRowFp8 = kRowBytesFp8 / 16;          // 65
constexpr int kHalfRowsFp8 = kWarpTokens * kRowBytesFp8;  // 8320 B: a token half's rows
constexpr int kHalfThreads = kThreads / 2;                // 128
// Three splits in flight per token half: against two, the 8-unit launch at
// 256K 54.2 -> 51.3-52.5 us and the 12-layer FP8 step 0.835 -> 0.798 ms
// (same box); four measured no faster launch and a slower step.
#ifndef QSA_ATTN_STAGES_FP8
#define QSA_ATTN_STAGES_FP8 3
#endif
#ifndef QSA_ATTN_HOST_CTAS_FP8
#define QSA_ATTN_HOST_CTAS_FP8 64
#endif
constexpr int kAStagesFp8 = QSA_ATTN_STAGES_FP8;          // splits in flight per half
constexpr int kMaxCtasHostFp8 = QSA_ATTN_HOST_CTAS_FP8;
constexpr int kSmemFp8 = 2 * kAStagesFp8 * kHalfRowsFp8;  // [half][stage][8][1040]
static_assert(kRowBytesFp8 % 16 == 0, "FP8 rows are whole 16-byte pieces");
static_assert(kAStagesFp8 >= 2, "a split is copied while the one before is computed");

// Four E4M3 codes (bytes of w, low first) -> four floats (exact).
__device__ __forceinline__ void e4m3x4_to_float4(uint32_t w, float& a, float& b, float& c, float& d) {
  uint32_t lo, hi;
  asm("{\n .reg .b16 x, y;\n mov.b32 {x, y}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, x;\n cvt.rn.f16x2.e4m3x2 %1, y;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
  const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  a = f0.x; b = f0.y; c = f1.x; d = f1.y;
}

// Row code (resolve_row) of token `tok` of the k-th split the CTA visits,
// and for a planned miss the hot row it goes to (else -1).
__device__ __forceinline__ int32_t row_code_fp8(const AttnParams& p, int u, int k, int split, int tok,
                                                int nsel, const int32_t* pend,
                                                const int32_t* pcode, const int32_t* pdst,
                                                int32_t* drow) {
  if (k < kPreSplits) {
    *drow = pdst[k * 16 + tok];
    return pcode[k * 16 + tok];
  }
  return resolve_row(p, u, split, tok, nsel, pend, drow);
}

// The 128 threads of token half `half` copy its 8 rows of the k-th split
// into rows ([8][1040]); absent rows are filled with zeros.
__device__ __forceinline__ void issue_rows_fp8(const AttnParams& p, int u, int k, int split, int nsel,
                                               int half, uint8_t* rows,
                                               const int32_t* pend, const int32_t* pcode,
                                               const int32_t* pdst) {
  const int t = threadIdx.x & (kHalfThreads - 1);
  for (int c = t; c < kWarpTokens * kChunksRowFp8; c += kHalfThreads) {
    const int i = c / kChunksRowFp8, off = c - i * kChunksRowFp8;
    int32_t drow;
    const int32_t code = row_code_fp8(p, u, k, split, half * kWarpTokens + i, nsel, pend, pcode, pdst,
                                      &drow);
    const uint8_t* src = row_ptr(p, u, code);
    cp_async16(rows + i * kRowBytesFp8 + off * 16, src ? src + off * 16 : p.b.pool, src ? 16u : 0u);
  }
}

// Planned misses of the k-th split: the half's threads copy the staged
// pieces they fetched into the misses' hot rows.
__device__ __forceinline__ void write_back_rows_fp8(const AttnParams& p, int u, int k, int split,
                                                    int nsel, int half,
                                                    const uint8_t* rows, const int32_t* pend,
                                                    const int32_t* pcode, const int32_t* pdst) {
  const int t = threadIdx.x & (kHalfThreads - 1);
  for (int c = t; c < kWarpTokens * kChunksRowFp8; c += kHalfThreads) {
    const int i = c / kChunksRowFp8, off = c - i * kChunksRowFp8;
    int32_t drow;
    row_code_fp8(p, u, k, split, half * kWarpTokens + i, nsel, pend, pcode, pdst, &drow);
    if (drow >= 0)
      *reinterpret_cast<uint4*>(p.b.pool + (int64_t)drow * p.b.row_bytes + off * 16) =
          *reinterpret_cast<const uint4*>(rows + i * kRowBytesFp8 + off * 16);
  }
}

// Barrier of the 128 threads of one token half (named barriers 1 and 2).
__device__ __forceinline__ void half_barrier(int half) {
  if (half == 0)
    asm volatile("bar.sync 1, %0;" ::"n"(kHalfThreads) : "memory");
  else
    asm volatile("bar.sync 2, %0;" ::"n"(kHalfThreads) : "memory");
}

__global__ void __maxnreg__(QSA_ATTN_MAXREG) attn_split_fp8_kernel(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];  // [half][stage][8][1040]
  __shared__ float xm[kKvHeads][kGroup], xl[kKvHeads][kGroup];
  __shared__ int32_t pre_code[kPreRows], pre_dst[kPreRows];
  __shared__ __align__(16) float xacc[kKvHeads][kGroup][kHeadDim];

  int u, r, cpu;
  cta_unit(p, blockIdx.x, u, r, cpu);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = warp & 3, half = warp >> 2;
  uint8_t* hbuf = smem + half * kAStagesFp8 * kHalfRowsFp8;
  grid_dependency_wait();   // the selection is read from here on
  int nsel = p.n_sel[u];
  if (nsel < 0 || nsel > p.k_max) {
    if (r == 0 && threadIdx.x == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernAttn, nsel);
    nsel = 0;
  }
  const int splits = (nsel + kBlocksPerSplit - 1) / kBlocksPerSplit;
  const int count = r < splits ? (splits - 1 - r) / cpu + 1 : 0;

  float qr[kGroup][4];
  {
    const uint16_t* qu = p.q + (int64_t)u * kQHeads * kHeadDim;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const uint2 w2 = *reinterpret_cast<const uint2*>(qu + (g * kGroup + j) * kHeadDim + 4 * lane);
      qr[j][0] = bf16_lo(w2.x) * p.scale_log2;
      qr[j][1] = bf16_hi(w2.x) * p.scale_log2;
      qr[j][2] = bf16_lo(w2.y) * p.scale_log2;
      qr[j][3] = bf16_hi(w2.y) * p.scale_log2;
    }
  }
  const int hj = (lane >> 3) & 3;
  float m_run = -INFINITY, l_run = 0.f;
  float acc[kGroup][4];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  const int32_t* pend = pending_map(p, u);
  preload_rows(p, u, r, cpu, count, nsel, pend, pre_code, pre_dst);
  // splits k + 1 .. k + kAStagesFp8 - 1 are in flight while split k is computed
#pragma unroll
  for (int k = 0; k < kAStagesFp8 - 1; ++k) {
    if (k < count)
      issue_rows_fp8(p, u, k, visit_split(k, count, r, cpu), nsel, half,
                     hbuf + k * kHalfRowsFp8, pend, pre_code, pre_dst);
    cp_async_commit();
  }
  for (int k = 0; k < count; ++k) {
    const int split = visit_split(k, count, r, cpu);
    cp_async_wait<kAStagesFp8 - 2>();   // this thread's pieces of split k have landed
    half_barrier(half);                 // everyone's have; split k - 1's stage is free
    const int kn = k + kAStagesFp8 - 1;
    if (kn < count)
      issue_rows_fp8(p, u, kn, visit_split(kn, count, r, cpu), nsel, half,
                     hbuf + (kn % kAStagesFp8) * kHalfRowsFp8, pend, pre_code, pre_dst);
    cp_async_commit();
    const uint8_t* R = hbuf + (k % kAStagesFp8) * kHalfRowsFp8;
    if (pend) write_back_rows_fp8(p, u, k, split, nsel, half, R, pend, pre_code, pre_dst);
    uint32_t valid_cur;
    {
      int32_t drow;
      const int32_t code = lane < kWarpTokens
                               ? row_code_fp8(p, u, k, split, half * kWarpTokens + lane, nsel, pend,
                                              pre_code, pre_dst, &drow)
                               : -1;
      valid_cur = __ballot_sync(0xFFFFFFFFu, code != -1) & ((1u << kWarpTokens) - 1u);
    }

    float x0 = -INFINITY;
#pragma unroll
    for (int i = 0; i < kWarpTokens; ++i) {
      const uint8_t* row = R + i * kRowBytesFp8;
      float k0, k1, k2, k3;
      e4m3x4_to_float4(*reinterpret_cast<const uint32_t*>(row + g * kHeadDim + 4 * lane), k0, k1, k2, k3);
      float d[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j)
        d[j] = fmaf(qr[j][3], k3, fmaf(qr[j][2], k2, fmaf(qr[j][1], k1, qr[j][0] * k0)));
      const bool up16 = lane & 16;
      const float a0 = up16 ? d[0] : d[2], a1 = up16 ? d[1] : d[3];
      const float r0 = __shfl_xor_sync(0xFFFFFFFFu, a0, 16);
      const float r1 = __shfl_xor_sync(0xFFFFFFFFu, a1, 16);
      const float v0 = (up16 ? d[2] : d[0]) + r0;
      const float v1 = (up16 ? d[3] : d[1]) + r1;
      const bool up8 = lane & 8;
      const float a = up8 ? v0 : v1;
      float v = (up8 ? v1 : v0) + __shfl_xor_sync(0xFFFFFFFFu, a, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
      const float ks = __half2float(*reinterpret_cast<const __half*>(row + 2 * kKvHeads * kHeadDim + 2 * g));
      if ((lane & 7) == i) x0 = ((valid_cur >> i) & 1u) ? v * ks : -INFINITY;
    }

    float ms = x0;
    ms = fmaxf(ms, __shfl_xor_sync(0xFFFFFFFFu, ms, 1));
    ms = fmaxf(ms, __shfl_xor_sync(0xFFFFFFFFu, ms, 2));
    ms = fmaxf(ms, __shfl_xor_sync(0xFFFFFFFFu, ms, 4));
    const float m_new = fmaxf(m_run, ms);
    const float so = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
    const float p0 = (x0 == -INFINITY) ? 0.f : exp2f(x0 - m_new);
    float ps = p0;
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 1);
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 2);
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 4);
    l_run = fmaf(l_run, so, ps);
    m_run = m_new;

#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const float sj = __shfl_sync(0xFFFFFFFFu, so, 8 * j);
      acc[j][0] *= sj; acc[j][1] *= sj; acc[j][2] *= sj; acc[j][3] *= sj;
    }
#pragma unroll
    for (int i = 0; i < kWarpTokens; ++i) {
      const uint8_t* row = R + i * kRowBytesFp8;
      float v0, v1, v2, v3;
      e4m3x4_to_float4(*reinterpret_cast<const uint32_t*>(row + kKvHeads * kHeadDim + g * kHeadDim + 4 * lane),
                       v0, v1, v2, v3);
      const float vs = __half2float(
          *reinterpret_cast<const __half*>(row + 2 * kKvHeads * kHeadDim + 2 * (kKvHeads + g)));
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const float pj = __shfl_sync(0xFFFFFFFFu, p0, 8 * j + i) * vs;
        acc[j][0] = fmaf(pj, v0, acc[j][0]);
        acc[j][1] = fmaf(pj, v1, acc[j][1]);
        acc[j][2] = fmaf(pj, v2, acc[j][2]);
        acc[j][3] = fmaf(pj, v3, acc[j][3]);
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  finish_split(p, u, r, g, half, lane, hj, m_run, l_run, acc, xm, xl, xacc);
  trigger_dependents();
}

// Merge: CTA (head, unit) of kMergeThreads threads.  The unit has cpu
// partials (up to QSA_MAX_BUDGET_TOKENS / 16 = 512).  Thread s reads the
// statistics of partial s; block reductions give the maximum M and the
// total L = sum_s 2^(m_s - M) l_s, and the weights 2^(m_s - M) go to shared
// memory.  Then kMergeGroups groups of 128 threads (one per output dim)
// each sum every kMergeGroups-th partial, and the groups' sums are added.
// A unit read from HBM alone can have 128 or more partials; one thread per
// dim walking all of them one dependent load after another took several
// microseconds.
constexpr int kMergeGroups = 4;
constexpr int kMergeThreads = kHeadDim * kMergeGroups;   // 512
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMaxPartials = QSA_MAX_BUDGET_TOKENS / (4 * kBlocksPerSplit);
static_assert(kMaxPartials <= kMergeThreads, "one partial per thread in the statistics pass");

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p) {
  grid_dependency_wait();
#if QSA_PDL_TRIGGER_MERGE
  trigger_dependents();
#endif
  __shared__ float wgt[kMaxPartials];
  __shared__ float red[kMergeWarps];
  __shared__ __align__(16) float part_acc[kMergeGroups][kHeadDim];
  const int h = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  int cpu = p.cta_start[u + 1] - p.cta_start[u];
  if (cpu > kMaxPartials) cpu = kMaxPartials;   // the launcher never grants more

  const float* ps = tid < cpu ? partial_ptr(p.b, u, tid) : nullptr;
  const float ms = ps ? ps[h] : -INFINITY;
  const float ls = ps ? ps[kQHeads + h] : 0.f;
  float v = ms;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float Mx = red[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) Mx = fmaxf(Mx, red[w]);
  const float ws = (ms == -INFINITY) ? 0.f : exp2f(ms - Mx);
  if (tid < cpu) wgt[tid] = ws;
  float lt = ws * ls;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(0xFFFFFFFFu, lt, o);
  __syncthreads();   // every warp has read red[] as maxima
  if (lane == 0) red[warp] = lt;
  __syncthreads();
  float Lt = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Lt += red[w];

  const int d = tid % kHeadDim, grp = tid / kHeadDim;
  float acc = 0.f;
  if (Mx != -INFINITY) {
#pragma unroll 8
    for (int s = grp; s < cpu; s += kMergeGroups)
      acc = fmaf(wgt[s], partial_ptr(p.b, u, s)[2 * kQHeads + h * kHeadDim + d], acc);
  }
  part_acc[grp][d] = acc;
  __syncthreads();
  if (grp == 0) {
    float a = part_acc[0][d];
#pragma unroll
    for (int g2 = 1; g2 < kMergeGroups; ++g2) a += part_acc[g2][d];
    float* o = p.out + ((int64_t)u * kQHeads + h) * kHeadDim;
    o[d] = Lt > 0.f ? a / Lt : 0.f;
    // the planned misses of the unit are in their hot rows now
    if (h == 0 && d == 0 && !p.gathered && p.b.hot_pend_on && p.b.u[u].hot_base >= 0)
      p.b.hot_pend_on[p.b.unit_state(u)] = 0;
    if (p.lse && d == 0)
      p.lse[(int64_t)u * kQHeads + h] = Lt > 0.f ? (Mx + log2f(Lt)) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_sparse_attn(const BatchDesc& b, const uint16_t* q, const int32_t* sel_blocks,
                               const int32_t* n_sel, int32_t budget_tokens,
                               const uint8_t* gathered, float softmax_scale, float* out,
                               float* lse, cudaStream_t s) {
  static PerDeviceOnce setup;
  cudaError_t e0 = setup.run([] {
    cudaError_t e = prefer_max_shared(attn_split_kernel, kSmemBytes);
    if (e == cudaSuccess) e = prefer_max_shared(attn_split_fp8_kernel, kSmemFp8);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_merge_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    return e;
  });
  int sm_count = 0;
  if (e0 == cudaSuccess) e0 = current_sm_count(&sm_count);
  if (e0 != cudaSuccess) return e0;
  AttnParams p;
  p.b = b;
  p.q = q;
  p.sel = sel_blocks;
  p.n_sel = n_sel;
  p.k_max = budget_tokens / 4;
  p.budget_tokens = budget_tokens;
  p.gathered = gathered;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = out;
  p.lse = lse;
  // Units that read host memory (units with hot rows read HBM only once
  // qsa_hot_cache_fetch has run) share the host cap; the others share the
  // remaining SMs.  A unit never gets more CTAs than splits or than the
  // workspace's partial slots.
  const int splits = (p.k_max + kBlocksPerSplit - 1) / kBlocksPerSplit;
  const bool fp8 = b.row_bytes == kRowBytesFp8;
  const int host_cap = fp8 ? kMaxCtasHostFp8 : kMaxCtasHost;
  int n_host = 0;
  for (int u = 0; u < b.n_units; ++u)
    n_host += gathered == nullptr && b.u[u].host_rows != nullptr && b.u[u].hot_base < 0;
  const int n_hbm = b.n_units - n_host;
  int cpu_max = splits < b.splits_max ? splits : b.splits_max;
  if (cpu_max < 1) cpu_max = 1;
  auto clamp = [&](int c) { return c < 1 ? 1 : (c > cpu_max ? cpu_max : c); };
  const int cpu_host = n_host ? clamp(host_cap / n_host) : 0;
  const int cpu_hbm = n_hbm ? clamp((kHbmCtasPerSm * sm_count - n_host * cpu_host) / n_hbm) : 0;
  int total = 0;
  for (int u = 0; u < b.n_units; ++u) {
    p.cta_start[u] = total;
    total += gathered == nullptr && b.u[u].host_rows != nullptr && b.u[u].hot_base < 0 ? cpu_host : cpu_hbm;
  }
  p.cta_start[b.n_units] = total;
  const int prio = highest_priority();
  cudaError_t e = fp8 ? launch_kernel(attn_split_fp8_kernel, dim3(total), dim3(kThreads), kSmemFp8,
                                      s, prio, dim3(1), p)
                      : launch_kernel(attn_split_kernel, dim3(total), dim3(kThreads), kSmemBytes,
                                      s, prio, dim3(1), p);
  if (e != cudaSuccess) return e;
  return launch_kernel(attn_merge_kernel, dim3(kQHeads, b.n_units), dim3(kMergeThreads), 0, s, prio,
                       dim3(1), p);
}

}  // namespace qsa
