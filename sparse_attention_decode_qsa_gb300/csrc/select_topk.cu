// Step 2 of the QSA decode step: per unit, keep the K = min(budget/4, #blocks)
// best C4 blocks under (score descending, block id ascending) and list them
// in ascending block id.  Each QSA layer selects on its own
// ("双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测", opening explanation of
// QSA); the budget is indexer_budget tokens ("Оффлоадинг KV-кэша
// Qwen3.8-Flash-Next в RAM через vLLM без потери скорости декодирования",
// lead paragraph).
//
// Method: radix select on order-preserving 32-bit keys, 8 bits per pass, to
// find the key T of the K-th best block and how many blocks equal to T must
// be kept; then one stable compaction in id order keeps every block above T
// and the first (lowest-id) blocks equal to T.  The compaction order gives the
// ascending-id output directly, and the tie rule falls out of it.  One CTA of
// 1024 threads per unit; the block scores were just written by the indexer
// and are read from L2.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

struct TopkParams {
  BatchDesc b;
  const float* blk;
  int64_t blk_stride;
  int32_t k_max;  // budget_tokens / 4
  int32_t* sel;   // [units][k_max]
  int32_t* n_sel; // [units]
};

// Larger float -> larger unsigned key; -0.0 is folded onto +0.0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t x = __float_as_uint(f);
  if (x == 0x80000000u) x = 0u;
  return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads) select_topk_kernel(const TopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_digit, s_krem;
  __shared__ uint32_t warp_gt[kWarps], warp_eq[kWarps];
  __shared__ uint32_t s_tot_gt, s_tot_eq;

  const int u = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t nb = (p.b.u[u].n + 3) / 4;
  const int K = nb < (int64_t)p.k_max ? (int)nb : p.k_max;
  const float* s = p.blk + (int64_t)u * p.blk_stride;
  int32_t* sel = p.sel + (int64_t)u * p.k_max;
  if (tid == 0) p.n_sel[u] = K;

  if (K == nb) {  // the budget covers the whole context: dense path
    for (int i = tid; i < K; i += kThreads) sel[i] = i;
    return;
  }

  // ---- radix select: T = key of the K-th largest, krem = ties to keep
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)K;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t i = tid; i < nb; i += kThreads) {
      const uint32_t k = order_key(s[i]);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255-8l .. 248-8l (top down)
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = hist[255 - 8 * lane - j]; sum += c[j]; }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - sum;
      if (excl < krem && krem <= incl) {
        uint32_t cum = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum + c[j] >= krem) { s_digit = 255u - 8u * lane - j; s_krem = krem - cum; break; }
          cum += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 0xFFu << shift;
    krem = s_krem;
    __syncthreads();
  }
  const uint32_t T = prefix;

  // ---- stable compaction in id order
  uint32_t out_base = 0, eq_base = 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t c0 = 0; c0 < nb; c0 += kThreads) {
    const int64_t i = c0 + tid;
    const uint32_t k = (i < nb) ? order_key(s[i]) : 0u;
    const bool gt = (i < nb) && k > T;
    const bool eq = (i < nb) && k == T;
    const uint32_t bg = __ballot_sync(0xFFFFFFFFu, gt), be = __ballot_sync(0xFFFFFFFFu, eq);
    if (lane == 0) { warp_gt[warp] = __popc(bg); warp_eq[warp] = __popc(be); }
    __syncthreads();
    if (warp == 0) {
      const uint32_t g = warp_gt[lane], e = warp_eq[lane];
      uint32_t ig = g, ie = e;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t vg = __shfl_up_sync(0xFFFFFFFFu, ig, o);
        const uint32_t ve = __shfl_up_sync(0xFFFFFFFFu, ie, o);
        if (lane >= o) { ig += vg; ie += ve; }
      }
      warp_gt[lane] = ig - g;
      warp_eq[lane] = ie - e;
      if (lane == 31) { s_tot_gt = ig; s_tot_eq = ie; }
    }
    __syncthreads();
    const uint32_t gt_excl = warp_gt[warp] + __popc(bg & lt_mask);
    const uint32_t eq_excl = warp_eq[warp] + __popc(be & lt_mask);
    const uint32_t remaining = krem > eq_base ? krem - eq_base : 0u;
    const bool take = gt || (eq && eq_excl < remaining);
    const uint32_t pos = out_base + gt_excl + min(eq_excl, remaining);
    if (take && pos < (uint32_t)K) sel[pos] = (int32_t)i;
    const uint32_t tot_gt = s_tot_gt, tot_eq = s_tot_eq;
    out_base += tot_gt + min(tot_eq, remaining);
    eq_base += tot_eq;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_select_topk(const BatchDesc& b, const float* blk_scores, int64_t blk_stride,
                               int32_t k_max, int32_t* sel_blocks, int32_t* n_sel,
                               cudaStream_t s) {
  TopkParams p;
  p.b = b;
  p.blk = blk_scores;
  p.blk_stride = blk_stride;
  p.k_max = k_max;
  p.sel = sel_blocks;
  p.n_sel = n_sel;
  select_topk_kernel<<<b.n_units, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
