// Step 2 of the QSA decode step: per unit, keep the K = min(budget/4, #blocks)
// best C4 blocks under (score descending, block id ascending) and list them
// in ascending block id.  Each QSA layer selects on its own
// ("双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测", opening explanation of
// QSA); the budget is indexer_budget tokens ("Оффлоадинг KV-кэша
// Qwen3.8-Flash-Next в RAM через vLLM без потери скорости декодирования",
// lead paragraph).
//
// Method: radix select on order-preserving 32-bit keys, digit by digit, to
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


// ---------------------------------------------------------------------------
// Cluster version: a cluster of kClusterCtas CTAs per unit.  CTA r keeps the
// keys of its slice [r*S, (r+1)*S) of the unit's blocks in shared memory, so
// the three radix passes (11, 11 and 10 bits) read no global memory.  Each
// pass builds a local histogram, then every CTA sums all CTAs' histograms
// through distributed shared memory and finds the threshold digit itself
// (all CTAs reach the same answer).  The compaction exchanges per-CTA counts
// of blocks above and equal to the threshold the same way, so every CTA
// writes its selected ids at their global ascending-id positions.
constexpr int kClusterCtas = 8;
constexpr int kMaxSlice = 32768;  // keys per CTA: 8 x 32768 blocks = 1M tokens
constexpr int kBins = 2048;
constexpr int kClusterSmem = kMaxSlice * 4;

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(p), out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(rank));
  return out;
}
__device__ __forceinline__ uint32_t ld_dsmem(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) select_topk_cluster_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t keys[];  // [kMaxSlice]
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t tot[kBins];
  __shared__ uint32_t warp_sum[kWarps];
  __shared__ uint32_t s_digit, s_krem;
  __shared__ uint32_t s_cnt[2];
  __shared__ uint32_t warp_gt[kWarps], warp_eq[kWarps];
  __shared__ uint32_t s_tot_gt, s_tot_eq;

  const uint32_t rank = cluster_rank();
  const int u = blockIdx.x / kClusterCtas;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nb = (p.b.u[u].n + 3) / 4;
  const int K = nb < (int64_t)p.k_max ? (int)nb : p.k_max;
  const float* s = p.blk + (int64_t)u * p.blk_stride;
  int32_t* sel = p.sel + (int64_t)u * p.k_max;
  const int64_t S = (nb + kClusterCtas - 1) / kClusterCtas;
  const int64_t lo = (int64_t)rank * S;
  const int64_t hi = lo + S < nb ? lo + S : nb;
  const int cnt = hi > lo ? (int)(hi - lo) : 0;
  if (rank == 0 && tid == 0) p.n_sel[u] = K;

  if (K == nb) {  // dense path: every block, in order
    for (int i = tid; i < cnt; i += kThreads) sel[lo + i] = (int32_t)(lo + i);
    return;       // uniform across the cluster: no DSMEM access follows
  }

  for (int i = tid; i < cnt; i += kThreads) keys[i] = order_key(s[lo + i]);

  uint32_t prefix = 0, mask = 0, krem = (uint32_t)K;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);  // digits of 11, 11, 10 bits
    const uint32_t nbins = pass == 2 ? 1024u : 2048u;
    if (pass > 0) cluster_wait();            // every CTA finished reading my hist
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < cnt; i += kThreads) {
      const uint32_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & (nbins - 1)], 1u);
    }
    __syncthreads();
    cluster_arrive();
    cluster_wait();                           // all histograms complete
    for (int b = tid; b < (int)nbins; b += kThreads) {
      uint32_t t = 0;
#pragma unroll
      for (int c = 0; c < kClusterCtas; ++c) t += ld_dsmem(dsmem_addr(&hist[b], c));
      tot[b] = t;
    }
    cluster_arrive();                         // done reading the others' hist
    __syncthreads();
    // threshold digit: scan bins from the top; warp w owns nbins/32 bins
    const int per = (int)nbins / kWarps;      // 64 or 32
    {
      uint32_t sum = 0;
      for (int j = lane; j < per; j += 32) sum += tot[nbins - 1 - (warp * per + j)];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      if (lane == 0) warp_sum[warp] = sum;
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t ws = warp_sum[lane];
      uint32_t incl = ws;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - ws;
      const bool mine = excl < krem && krem <= incl;
      const uint32_t owners = __ballot_sync(0xFFFFFFFFu, mine);
      const uint32_t owner = owners ? (uint32_t)(__ffs(owners) - 1) : 0u;  // always one by construction
      const uint32_t base = __shfl_sync(0xFFFFFFFFu, excl, owner);
      // owner warp range, bins from the top: index j -> bin nbins-1-(owner*per+j)
      uint32_t cum = base;
      for (int j0 = 0; j0 < per; j0 += 32) {
        const uint32_t c = tot[nbins - 1 - (owner * per + j0 + lane)];
        uint32_t ic = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, ic, o);
          if (lane >= o) ic += v;
        }
        const uint32_t ex = cum + ic - c;
        const bool hit = ex < krem && krem <= cum + ic;
        const uint32_t hb = __ballot_sync(0xFFFFFFFFu, hit);
        if (hb) {
          const int hl = __ffs(hb) - 1;
          if (lane == hl) {
            s_digit = nbins - 1 - (owner * per + j0 + hl);
            s_krem = krem - ex;
          }
          break;
        }
        cum += __shfl_sync(0xFFFFFFFFu, ic, 31);
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= (nbins - 1) << shift;
    krem = s_krem;
  }
  const uint32_t T = prefix;

  // ---- per-CTA counts above / equal to T, exchanged through DSMEM
  {
    uint32_t g = 0, e = 0;
    for (int i = tid; i < cnt; i += kThreads) {
      g += keys[i] > T;
      e += keys[i] == T;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xFFFFFFFFu, g, o);
      e += __shfl_xor_sync(0xFFFFFFFFu, e, o);
    }
    if (lane == 0) { warp_gt[warp] = g; warp_eq[warp] = e; }
    cluster_wait();                           // pass-2 readers of hist are done (s_cnt is separate)
    __syncthreads();
    if (tid == 0) {
      uint32_t tg = 0, te = 0;
      for (int w = 0; w < kWarps; ++w) { tg += warp_gt[w]; te += warp_eq[w]; }
      s_cnt[0] = tg;
      s_cnt[1] = te;
    }
    __syncthreads();
  }
  cluster_arrive();
  cluster_wait();
  uint32_t base_gt = 0, base_eq = 0;
  for (uint32_t c = 0; c < rank; ++c) {
    base_gt += ld_dsmem(dsmem_addr(&s_cnt[0], c));
    base_eq += ld_dsmem(dsmem_addr(&s_cnt[1], c));
  }

  // ---- stable compaction of this slice in id order
  uint32_t out_base = base_gt, eq_base = base_eq;  // counts before this chunk, globally
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < cnt; c0 += kThreads) {
    const int i = c0 + tid;
    const uint32_t k = i < cnt ? keys[i] : 0u;
    const bool gt = i < cnt && k > T;
    const bool eq = i < cnt && k == T;
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
    const uint32_t gt_before = out_base + warp_gt[warp] + __popc(bg & lt_mask);
    const uint32_t eq_before = eq_base + warp_eq[warp] + __popc(be & lt_mask);
    const bool take = gt || (eq && eq_before < krem);
    const uint32_t pos = gt_before + min(eq_before, krem);
    if (take && pos < (uint32_t)K) sel[pos] = (int32_t)(lo + i);
    out_base += s_tot_gt;
    eq_base += s_tot_eq;
    __syncthreads();
  }
  cluster_arrive();                            // keep s_cnt alive until every CTA read it
  cluster_wait();
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
  int64_t nb_max = 0;
  for (int u = 0; u < b.n_units; ++u) {
    const int64_t nb = (b.u[u].n + 3) / 4;
    if (nb > nb_max) nb_max = nb;
  }
  if (nb_max > (int64_t)kClusterCtas * kMaxSlice) {  // beyond 1M tokens: one CTA per unit
    select_topk_kernel<<<b.n_units, kThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = prefer_max_shared(select_topk_cluster_kernel, kClusterSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(b.n_units * kClusterCtas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kClusterSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_topk_cluster_kernel, p);
}

}  // namespace qsa
