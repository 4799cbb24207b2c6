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
// ascending-id output directly, and the tie rule falls out of it.  Units of
// up to 1M tokens use a cluster of 8 CTAs (below); longer ones one CTA of
// 1024 threads.  The block scores were just written by the indexer and are
// read from L2.
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
  grid_dependency_wait();
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
// Cluster version: a cluster of kClusterCtas CTAs of 512 threads per unit.
// CTA r keeps the keys of its slice [r*S, (r+1)*S) of the unit's blocks in
// shared memory.  The first digit (the top 11 bits of the key) comes from a
// histogram that every CTA adds into every CTA's total with remote atomic
// adds (block scores crowd into a few exponent bins, so few bins are
// non-zero).  If the boundary bin holds at most kCandMax keys and no CTA
// more than kRegion of them - the usual case - every CTA sends its keys in
// that bin, and its counts of keys in and above it, to every CTA; each CTA
// then finds the threshold T among the candidates (one warp ranks them
// directly when they are at most 32, as for planted workloads, where the
// K-th score stands alone in its bin; else a radix select of 11 and 10
// bits) and knows every CTA's counts of keys above and equal to T, so it
// writes its selected ids at their global ascending-id positions with no
// further exchange.  Otherwise two more cluster-wide passes over every key
// find T and the CTAs exchange their counts.  A CTA takes half an SM's
// registers, so it can share an SM with other kernels.
constexpr int kClusterCtas = 8;
static_assert(kClusterCtas <= 8, "cross-CTA sums reduce over lanes 0..7");
constexpr int kCThreads = 512;
constexpr int kCWarps = kCThreads / 32;
static_assert(kCWarps <= 32 && kClusterCtas <= 32, "per-warp and per-CTA counts are summed by one warp");
static_assert(kCThreads > kClusterCtas * 32, "warps beyond the first kClusterCtas credit the candidates");
constexpr int kMaxSlice = 32768;  // keys per CTA: 8 x 32768 blocks = 1M tokens
constexpr int kBins = 2048;
constexpr int kCandMax = 2048;    // boundary-bin keys the CTAs finish the select on
constexpr int kRegion = kCandMax / kClusterCtas;   // slots per source CTA in the candidate list
constexpr int kSubHists = 4;      // first-digit histogram copies (warps w % 4), less contention
static_assert(kCandMax * 8 <= kSubHists * kBins * 4, "candidates reuse the sub-histograms");

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
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
__device__ __forceinline__ void st_dsmem(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Digit of the krem-th largest key from a histogram of nbins bins (counted
// from the top; nbins 1024 or 2048): *digit, and *krem_out = its rank within
// that bin.  Thread t owns the bins nbins-1-per*t .. nbins-per*(t+1) (per =
// nbins / kCThreads, one vector load); a scan over the threads finds the one
// thread whose bins hold rank krem.  Called by the whole CTA; the results are
// valid after the closing __syncthreads().
static_assert(kCThreads * 4 == kBins && kCThreads * 2 == 1024, "find_digit: 4 or 2 bins per thread");
__device__ __forceinline__ void find_digit(const uint32_t* h, uint32_t nbins, uint32_t krem,
                                           uint32_t* warp_sum, uint32_t* digit,
                                           uint32_t* krem_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t c[4];   // c[j]: bin nbins-1-(per*t+j)
  int per;
  if (nbins == 2048u) {
    per = 4;
    const uint4 v = *reinterpret_cast<const uint4*>(h + 2048 - 4 * (tid + 1));
    c[0] = v.w; c[1] = v.z; c[2] = v.y; c[3] = v.x;
  } else {
    per = 2;
    const uint2 v = *reinterpret_cast<const uint2*>(h + 1024 - 2 * (tid + 1));
    c[0] = v.y; c[1] = v.x; c[2] = 0u; c[3] = 0u;
  }
  const uint32_t sum = c[0] + c[1] + c[2] + c[3];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  uint32_t cum = incl - sum;
  for (int w = 0; w < warp; ++w) cum += warp_sum[w];
  if (cum < krem && krem <= cum + sum) {   // exactly one thread when krem is in range
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < per && cum + c[j] >= krem) {
        *digit = nbins - 1u - (uint32_t)(per * tid + j);
        *krem_out = krem - cum;
        break;
      }
      cum += c[j];
    }
  }
  __syncthreads();
}

// red.shared::cluster: add v to a shared variable of another CTA of the cluster.
__device__ __forceinline__ void red_dsmem(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// 40 registers x 512 threads: a CTA fits on an SM beside two index-score CTAs.
__global__ void __maxnreg__(40) select_topk_cluster_kernel(const TopkParams p, int slice_cap) {
  extern __shared__ __align__(16) uint32_t dyn[];
  uint32_t* keys = dyn;                                   // [slice_cap]
  uint32_t* sub = dyn + slice_cap;                        // [kSubHists][kBins], first digit
  // later the same space holds the unit's boundary-bin candidates (all CTAs')
  uint32_t* cand_key = sub;                               // [kCandMax]: low 21 bits
  __shared__ __align__(16) uint32_t hist[kBins];         // this CTA's first-digit histogram
  __shared__ __align__(16) uint32_t tot[kBins];          // the unit's, summed over the cluster
  __shared__ uint32_t warp_sum[kCWarps];
  __shared__ uint32_t s_digit, s_krem, s_pos, s_above;
  __shared__ uint32_t s_cnt[2];
  __shared__ uint32_t c_bin[kClusterCtas], c_above[kClusterCtas];   // per CTA: keys in / above bin d1
  __shared__ uint32_t c_gt[kClusterCtas], c_eq[kClusterCtas];       // per CTA: keys above / equal to T
  __shared__ uint32_t warp_gt[kCWarps], warp_eq[kCWarps];
  __shared__ uint32_t cand_idx[kRegion];                            // slice index of my candidates

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

  // the histograms are zeroed before the wait for the kernel before this
  // one (shared memory only), so that work overlaps its tail
  if (K != nb) {
    for (int i = tid; i < kBins; i += kCThreads) tot[i] = 0;
    for (int i = tid; i < kSubHists * kBins; i += kCThreads) sub[i] = 0;
    if (tid == 0) { s_pos = 0; s_above = 0; }
  }
  __syncthreads();
  grid_dependency_wait();
  if (rank == 0 && tid == 0) p.n_sel[u] = K;

  if (K == nb) {  // dense path: every block, in order
    for (int i = tid; i < cnt; i += kCThreads) sel[lo + i] = (int32_t)(lo + i);
    return;       // uniform across the cluster: no DSMEM access follows
  }
  cluster_arrive();   // my tot is zeroed (waited for once the keys are in)

  // ---- first digit: bits 31..21, counted into kSubHists copies while the
  // keys are loaded, then folded into hist
  {
    // kLoadBatch loads in flight per thread before their keys are counted.
    // (Counting with one atomic per distinct bin of a warp, lanes grouped by
    // __match_any_sync, was measured slower: 18.3 against 15.0 us per 8-unit
    // launch of 262144 tokens.)
    constexpr int kLoadBatch = 8;
    uint32_t* h = sub + (warp % kSubHists) * kBins;
    const float* src = s + lo;
    int done = 0;   // keys loaded by the vector path below
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      // four keys per 16-byte load, kLoadBatch / 2 loads in flight per thread
      constexpr int kVec = kLoadBatch / 2;
      const int n4 = cnt / 4;
      const float4* src4 = reinterpret_cast<const float4*>(src);
      for (int j0 = tid; j0 < n4; j0 += kCThreads * kVec) {
        float4 v[kVec];
#pragma unroll
        for (int b = 0; b < kVec; ++b) {
          const int j = j0 + b * kCThreads;
          v[b] = j < n4 ? __ldg(src4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < kVec; ++b) {
          const int j = j0 + b * kCThreads;
          if (j < n4) {
            const uint4 k = make_uint4(order_key(v[b].x), order_key(v[b].y), order_key(v[b].z),
                                       order_key(v[b].w));
            *reinterpret_cast<uint4*>(keys + 4 * j) = k;
            atomicAdd(&h[k.x >> 21], 1u);
            atomicAdd(&h[k.y >> 21], 1u);
            atomicAdd(&h[k.z >> 21], 1u);
            atomicAdd(&h[k.w >> 21], 1u);
          }
        }
      }
      done = 4 * n4;
    }
    for (int i0 = done + tid; i0 < cnt; i0 += kCThreads * kLoadBatch) {
      float v[kLoadBatch];
#pragma unroll
      for (int j = 0; j < kLoadBatch; ++j) {
        const int i = i0 + j * kCThreads;
        v[j] = i < cnt ? __ldg(s + lo + i) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kLoadBatch; ++j) {
        const int i = i0 + j * kCThreads;
        if (i < cnt) {
          const uint32_t k = order_key(v[j]);
          keys[i] = k;
          atomicAdd(&h[k >> 21], 1u);
        }
      }
    }
  }
  __syncthreads();
  // The cluster's histogram: every CTA adds its non-zero bins (the sums of
  // its sub-histograms) into every CTA's tot (remote atomic adds, fire and
  // forget; block scores crowd into few bins), so each CTA then holds the
  // sum locally.  The sub-histograms are read here for the last time: the
  // candidates that later land in the same space come after the barrier.
  cluster_wait();                              // every CTA's tot is zeroed
  for (int b = tid; b < kBins; b += kCThreads) {
    uint32_t v = 0;
#pragma unroll
    for (int c = 0; c < kSubHists; ++c) v += sub[c * kBins + b];
    if (v) {
#pragma unroll
      for (int c = 0; c < kClusterCtas; ++c) red_dsmem(dsmem_addr(&tot[b], (uint32_t)c), v);
    }
  }
  cluster_sync();                              // every tot holds the unit's histogram
  find_digit(tot, kBins, (uint32_t)K, warp_sum, &s_digit, &s_krem);
  const uint32_t d1 = s_digit;
  uint32_t krem = s_krem;
  uint32_t T;
  // warp w owns the contiguous keys [w*R, (w+1)*R) of the slice (R a multiple
  // of 128) in the walks below, lane l taking keys 4l .. 4l+3 of each step of
  // 128 (one 16-byte load)
  const int R = ((cnt + kCWarps - 1) / kCWarps + 127) / 128 * 128;
  const int w0 = warp * R, w1 = w0 + R < cnt ? w0 + R : cnt;
  const uint4* kw = reinterpret_cast<const uint4*>(keys);   // slice_cap is a multiple of 4
  bool fast = tot[d1] <= (uint32_t)kCandMax;
  if (fast) {
    // ---- usual path: every CTA sends its keys in bin d1 (low 21 bits) to
    // its own region of kRegion slots in every CTA's candidate list, and its
    // counts of keys in and above the bin to every CTA; each CTA then
    // finishes the select on the candidates alone and knows every CTA's
    // counts of keys above and equal to T, so no further cluster barrier is
    // needed.  A CTA with more than kRegion keys in the bin sends the first
    // kRegion; all CTAs see its count and take the general path below.
    // The walk is the compaction's (warp ranges), so each warp's count of
    // keys above the bin (all above T) comes with it, and the slice index
    // of each candidate is kept to credit it to its warp once T is known:
    // the usual path needs no separate counting walk.  A lane with keys in
    // the bin reserves their slots itself (they are few: one atomic per such
    // lane and step).
    uint32_t above = 0;
    for (int i0 = w0; i0 < w1; i0 += 128) {
      const int i = i0 + 4 * lane;
      const uint4 q = i < w1 ? kw[i / 4] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
      uint32_t hits = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = i + e < w1;
        hits |= (in && (kq[e] >> 21) == d1) ? (1u << e) : 0u;
        above += (in && (kq[e] >> 21) > d1) ? 1u : 0u;
      }
      if (hits) {
        uint32_t pos = atomicAdd(&s_pos, (uint32_t)__popc(hits));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (((hits >> e) & 1u) && pos < (uint32_t)kRegion) {
#pragma unroll
            for (int c = 0; c < kClusterCtas; ++c)
              st_dsmem(dsmem_addr(&cand_key[rank * kRegion + pos], (uint32_t)c), kq[e] & 0x1FFFFFu);
            cand_idx[pos] = (uint32_t)(i + e);
          }
          pos += (hits >> e) & 1u;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xFFFFFFFFu, above, o);
    if (lane == 0) {
      warp_gt[warp] = above;
      warp_eq[warp] = 0;
      if (above) atomicAdd(&s_above, above);
    }
    __syncthreads();
    if (warp == 0 && lane < kClusterCtas) {
      st_dsmem(dsmem_addr(&c_above[rank], (uint32_t)lane), s_above);
      st_dsmem(dsmem_addr(&c_bin[rank], (uint32_t)lane), s_pos);
    }
    cluster_sync();                            // every CTA holds all candidates and counts
    for (int c = 0; c < kClusterCtas; ++c) fast = fast && c_bin[c] <= (uint32_t)kRegion;
  }
  if (fast) {
    uint32_t prefix = 0;
    if (tot[d1] <= 32u) {
      // At most 32 keys in the bin (the usual case: the K-th block score
      // stands alone in its first-digit bin): every warp ranks them itself,
      // so no barrier is needed.  Lane i holds candidate i; its value is the
      // krem-th largest when fewer than krem candidates are greater and at
      // least krem are greater or equal.  krem then becomes the number of
      // keys equal to T that are taken (krem minus the candidates above T),
      // as after the radix passes.
      const uint32_t C = tot[d1];
      uint32_t cb[kClusterCtas];   // candidates per source CTA
#pragma unroll
      for (int c = 0; c < kClusterCtas; ++c) cb[c] = c_bin[c];
      const bool valid = (uint32_t)lane < C;
      uint32_t v = 0;
      if (valid) {
        uint32_t i = (uint32_t)lane, c = 0;
#pragma unroll
        for (int k = 0; k + 1 < kClusterCtas; ++k) {
          if (c == (uint32_t)k && i >= cb[k]) { i -= cb[k]; c = (uint32_t)k + 1; }
        }
        v = cand_key[c * kRegion + i];
      }
      uint32_t gt = 0, eq = 0;
      for (uint32_t j = 0; j < C; ++j) {
        const uint32_t vj = __shfl_sync(0xFFFFFFFFu, v, (int)j);
        gt += vj > v ? 1u : 0u;
        eq += vj == v ? 1u : 0u;
      }
      const uint32_t hit = __ballot_sync(0xFFFFFFFFu, valid && gt < krem && krem <= gt + eq);
      const int src = hit ? __ffs(hit) - 1 : 0;
      prefix = __shfl_sync(0xFFFFFFFFu, v, src);
      krem -= __shfl_sync(0xFFFFFFFFu, gt, src);
    } else {
      // two radix passes over the candidates (11 and 10 bits)
      uint32_t mask = 0;
      for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const uint32_t nbins = pass == 0 ? 2048u : 1024u;
        for (int i = tid; i < (int)nbins; i += kCThreads) hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < kCandMax; j += kCThreads) {
          const uint32_t k = cand_key[j];
          if ((uint32_t)(j % kRegion) < c_bin[j / kRegion] && (k & mask) == prefix)
            atomicAdd(&hist[(k >> shift) & (nbins - 1)], 1u);
        }
        __syncthreads();
        find_digit(hist, nbins, krem, warp_sum, &s_digit, &s_krem);
        prefix |= s_digit << shift;
        mask |= (nbins - 1) << shift;
        krem = s_krem;
        __syncthreads();
      }
    }
    T = (d1 << 21) | prefix;
    // warp c: CTA c's keys above T (above bin d1, or candidates above) and equal to T
    if (warp < kClusterCtas) {
      uint32_t g = 0, e = 0;
      for (uint32_t j = lane; j < c_bin[warp]; j += 32) {
        const uint32_t k = cand_key[warp * kRegion + j];
        g += k > prefix ? 1u : 0u;
        e += k == prefix ? 1u : 0u;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        g += __shfl_xor_sync(0xFFFFFFFFu, g, o);
        e += __shfl_xor_sync(0xFFFFFFFFu, e, o);
      }
      if (lane == 0) { c_gt[warp] = c_above[warp] + g; c_eq[warp] = e; }
    } else {
      // the other warps credit this CTA's candidates above / equal to T to
      // the warps whose ranges hold them
      constexpr uint32_t kFirst = kClusterCtas * 32, kStride = kCThreads - kClusterCtas * 32;
      for (uint32_t j = (uint32_t)tid - kFirst; j < c_bin[rank]; j += kStride) {
        const uint32_t k = cand_key[rank * kRegion + j];
        const int w = (int)cand_idx[j] / R;
        if (k > prefix) atomicAdd(&warp_gt[w], 1u);
        else if (k == prefix) atomicAdd(&warp_eq[w], 1u);
      }
    }
    __syncthreads();
  } else {
    // ---- general path: two more cluster-wide passes over every key
    uint32_t prefix = d1 << 21, mask = 0x7FFu << 21;
    for (int pass = 1; pass < 3; ++pass) {
      const int shift = pass == 1 ? 10 : 0;
      const uint32_t nbins = pass == 1 ? 2048u : 1024u;
      cluster_sync();                          // every CTA finished reading my hist
      for (int i = tid; i < kBins; i += kCThreads) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < cnt; i += kCThreads) {
        const uint32_t k = keys[i];
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & (nbins - 1)], 1u);
      }
      __syncthreads();
      cluster_sync();                          // all histograms complete
      for (int b = tid; b < (int)nbins; b += kCThreads) {
        uint32_t t = 0;
#pragma unroll
        for (int c = 0; c < kClusterCtas; ++c) t += ld_dsmem(dsmem_addr(&hist[b], c));
        tot[b] = t;
      }
      __syncthreads();
      find_digit(tot, nbins, krem, warp_sum, &s_digit, &s_krem);
      prefix |= s_digit << shift;
      mask |= (nbins - 1) << shift;
      krem = s_krem;
    }
    T = prefix;
  }

  // ---- compaction over the warp ranges.  Each warp's counts of keys above
  // / equal to T (from the candidate walk on the usual path, from a counting
  // walk otherwise), one warp sum of the lower warps' totals gives the
  // offsets within the CTA, and a second walk writes the selected ids in id
  // order (ballots per key position count the lower lanes' keys, only in
  // steps that select a key), after the keys of the lower-rank CTAs (known
  // locally on the usual path, exchanged through DSMEM otherwise).
  if (!fast) {
    uint32_t g = 0, e = 0;
    for (int i0 = w0; i0 < w1; i0 += 128) {
      const int i = i0 + 4 * lane;
      const uint4 q = i < w1 ? kw[i / 4] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        g += (i + x < w1 && kq[x] > T) ? 1u : 0u;
        e += (i + x < w1 && kq[x] == T) ? 1u : 0u;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xFFFFFFFFu, g, o);
      e += __shfl_xor_sync(0xFFFFFFFFu, e, o);
    }
    if (lane == 0) { warp_gt[warp] = g; warp_eq[warp] = e; }
    __syncthreads();
  }
  // keys above / equal to T before the warp's range, globally: lane i adds
  // the counts of warp i < warp (and, on the usual path, of CTA i < rank),
  // then the warp sums them
  uint32_t gt_run = 0, eq_run = 0;
  if (lane < warp) { gt_run = warp_gt[lane]; eq_run = warp_eq[lane]; }
  if (fast && (uint32_t)lane < rank) { gt_run += c_gt[lane]; eq_run += c_eq[lane]; }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt_run += __shfl_xor_sync(0xFFFFFFFFu, gt_run, o);
    eq_run += __shfl_xor_sync(0xFFFFFFFFu, eq_run, o);
  }
  if (!fast) {
    if (tid == 0) {
      uint32_t sg = 0, se = 0;
      for (int w = 0; w < kCWarps; ++w) { sg += warp_gt[w]; se += warp_eq[w]; }
      s_cnt[0] = sg;
      s_cnt[1] = se;
    }
    cluster_sync();                                        // every CTA's totals are published
    uint32_t vg = 0u, ve = 0u;   // lane c < rank reads CTA c's totals
    if ((uint32_t)lane < rank) {
      vg = ld_dsmem(dsmem_addr(&s_cnt[0], (uint32_t)lane));
      ve = ld_dsmem(dsmem_addr(&s_cnt[1], (uint32_t)lane));
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      vg += __shfl_xor_sync(0xFFFFFFFFu, vg, o);
      ve += __shfl_xor_sync(0xFFFFFFFFu, ve, o);
    }
    gt_run += __shfl_sync(0xFFFFFFFFu, vg, 0);   // lanes 0..7 hold the sums
    eq_run += __shfl_sync(0xFFFFFFFFu, ve, 0);
  }
  for (int i0 = w0; i0 < w1; i0 += 128) {
    const int i = i0 + 4 * lane;
    const uint4 q = i < w1 ? kw[i / 4] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
    uint32_t mg = 0, me = 0;   // this lane's keys above / equal to T
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      mg |= (i + x < w1 && kq[x] > T) ? (1u << x) : 0u;
      me |= (i + x < w1 && kq[x] == T) ? (1u << x) : 0u;
    }
    if (!__any_sync(0xFFFFFFFFu, (mg | me) != 0u)) continue;   // warp-uniform
    // keys of the lower lanes come first in id order: one ballot per key
    // position counts them, with no chain of dependent shuffles
    const uint32_t below = (1u << lane) - 1u;
    uint32_t gb = gt_run, eb = eq_run, tg = 0, te = 0;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const uint32_t bg = __ballot_sync(0xFFFFFFFFu, (mg >> x) & 1u);
      const uint32_t be = __ballot_sync(0xFFFFFFFFu, (me >> x) & 1u);
      gb += __popc(bg & below);
      eb += __popc(be & below);
      tg += __popc(bg);
      te += __popc(be);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      if ((mg >> x) & 1u) {
        const uint32_t pos = gb + min(eb, krem);
        if (pos < (uint32_t)K) sel[pos] = (int32_t)(lo + i + x);
        ++gb;
      } else if ((me >> x) & 1u) {
        if (eb < krem && gb + eb < (uint32_t)K) sel[gb + eb] = (int32_t)(lo + i + x);
        ++eb;
      }
    }
    gt_run += tg;
    eq_run += te;
  }
  trigger_dependents();
  if (!fast) cluster_sync();   // keep s_cnt alive until every CTA read it
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
    return launch_kernel(select_topk_kernel, dim3(b.n_units), dim3(kThreads), 0, s, 0, dim3(1), p);
  }
  constexpr int kMaxDynSmem = kMaxSlice * 4 + kSubHists * kBins * 4;
  static PerDeviceOnce setup;
  const cudaError_t e =
      setup.run([] { return prefer_max_shared(select_topk_cluster_kernel, kMaxDynSmem); });
  if (e != cudaSuccess) return e;
  // keys per CTA of the largest unit, rounded up to 16-byte multiples
  const int slice_cap = (int)(((nb_max + kClusterCtas - 1) / kClusterCtas + 3) / 4 * 4);
  return launch_kernel(select_topk_cluster_kernel, dim3(b.n_units * kClusterCtas), dim3(kCThreads),
                       (size_t)slice_cap * 4 + kSubHists * kBins * 4, s, 0, dim3(kClusterCtas), p,
                       slice_cap);
}

}  // namespace qsa
