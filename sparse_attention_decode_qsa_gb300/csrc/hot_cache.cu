// Cross-step hot cache of the QSA decode step ("双卡RTX4090跑通Qwen3-Next：
// 8并发满血长上下文实测", section "显存账本：热缓存卸载省下约84%": the full
// history stays in pinned host memory, missing blocks are moved back to the
// GPU on demand into a hot cache, and logical tokens are found through a slot
// table kept apart from the physical rows).
//
// Each offloaded (request, layer) owns H pool rows.  Per step, after top-k:
//   hot_plan_kernel  one CTA of 1024 threads per unit.  Marks the hot rows the
//                    selected tokens already hold (a shared-memory bitmask),
//                    ranks the cold selected tokens in ascending token order
//                    (block scan), ranks the rows not in use in circular
//                    order from the unit's cursor (second block scan), hands
//                    the r-th such row to the r-th miss, reads the rows'
//                    previous owners, then (after a barrier) writes the slot
//                    table, the owners, the cursor and a fill list
//                    {token, pool row} in the workspace.
//   hot_fill_kernel  copies each listed host row into its hot row: 8 rows
//                    per CTA, every 16-byte load of a thread issued before
//                    its stores.  Few rows per CTA spread a step's misses
//                    over many SMs: reads of host pages the GPU has not
//                    touched lately are slow (a cost per page, not per
//                    byte), and more SMs keep more of them in flight.
// Afterwards every selected row of the unit is in HBM.
// qsa_hot_cache_plan runs the plan alone and also writes, per selected
// position, the row its miss goes to: the next attention of the unit reads
// those rows from host memory (once, as a zero-copy read would) and writes
// them into their hot rows, so a miss costs no separate copy pass.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kMaxTokPerThread = QSA_MAX_BUDGET_TOKENS / kPlanThreads;   // 8
constexpr int kFillThreads = 256;
constexpr int kFillRows = 8;
// plan kernel shared memory at the limits: bitmask of QSA_MAX_HOT_ROWS rows +
// one victim per token of the largest budget
constexpr int kPlanSmemMax = QSA_MAX_HOT_ROWS / 8 + QSA_MAX_BUDGET_TOKENS * 4;
static_assert(kPlanSmemMax <= 48 * 1024, "plan kernel fits the default dynamic shared memory");
static_assert(QSA_MAX_BUDGET_TOKENS % kPlanThreads == 0, "tokens per thread");

struct HotParams {
  BatchDesc b;
  const int32_t* sel;
  const int32_t* n_sel;
  int32_t k_max;           // stride of sel (budget_tokens / 4)
  int32_t plan_only;       // 1: leave the copies to the next attention (pending map)
};

// Exclusive scan of v over the CTA; *total receives the sum.  Every thread
// of the CTA must call it (it holds three barriers; the last one lets the
// next call reuse s_warp).
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kPlanWarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kPlanWarps) s_warp[lane] = w;   // inclusive warp prefix
  }
  __syncthreads();
  *total = s_warp[kPlanWarps - 1];
  const int before = warp > 0 ? s_warp[warp - 1] : 0;
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kPlanThreads) hot_plan_kernel(const HotParams p) {
  grid_dependency_wait();
  extern __shared__ uint32_t in_use[];         // [ceil(H / 32)] bitmask, then victim[budget]
  __shared__ int s_warp[kPlanWarps];
  __shared__ int s_bad;
  const int u = blockIdx.x, tid = threadIdx.x;
  const int H = p.b.hot_rows;
  const int64_t hb = p.b.u[u].hot_base;
  const int64_t st = p.b.unit_state(u);
  if (hb < 0 || H <= 0) {
    if (tid == 0 && p.b.hot_nfill) p.b.hot_nfill[st] = 0;
    return;
  }
  const int64_t n = p.b.u[u].n;
  const int nsel = p.n_sel[u];
  if (nsel < 0 || nsel > p.k_max) {
    if (tid == 0) {
      report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernHot, nsel);
      p.b.hot_nfill[st] = 0;
      p.b.hot_pend_on[st] = 0;
    }
    return;
  }
  const int c0 = p.b.hot_cursor[st];   // read early: it overlaps the classification
  const int words = (H + 31) / 32;
  int32_t* victim = reinterpret_cast<int32_t*>(in_use + words);
  int32_t* slots = p.b.slot_table + p.b.unit_row(u);
  int32_t* owner = p.b.hot_owner + st * H;
  for (int i = tid; i < words; i += kPlanThreads) in_use[i] = 0u;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // ---- classify the selected tokens (thread tid: tokens j = tid*per .. +per-1)
  const int ntok = 4 * nsel;
  const int per = (ntok + kPlanThreads - 1) / kPlanThreads;   // <= kMaxTokPerThread
  int32_t tok[kMaxTokPerThread];
  int my_miss = 0;
#pragma unroll
  for (int i = 0; i < kMaxTokPerThread; ++i) {
    tok[i] = -1;
    const int j = tid * per + i;
    if (i >= per || j >= ntok) continue;
    const int64_t blk = p.sel[(int64_t)u * p.k_max + (j >> 2)];
    if (blk < 0 || 4 * blk >= n) {
      if ((j & 3) == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernHot, blk);
      s_bad = 1;
      continue;
    }
    const int64_t t = 4 * blk + (j & 3);
    if (t >= n) continue;
    const int32_t s = slots[t];
    if ((int64_t)s >= hb && (int64_t)s < hb + H) {
      const int v = (int)(s - hb);
      atomicOr(&in_use[v >> 5], 1u << (v & 31));
    } else if (s == -1) {
      tok[i] = (int32_t)t;
      ++my_miss;
    }
  }
  int m;
  const int miss_base = block_exclusive_scan(my_miss, &m, s_warp);
  if (s_bad) {                                   // uniform: written before the scan's barriers
    if (tid == 0) {
      p.b.hot_nfill[st] = 0;
      p.b.hot_pend_on[st] = 0;
    }
    return;
  }

  // ---- rows not in use, in circular order from the cursor
  const int cursor = (c0 >= 0 && c0 < H) ? c0 : 0;
  const int hper = (H + kPlanThreads - 1) / kPlanThreads;
  int my_free = 0;
  for (int i = 0; i < hper; ++i) {
    const int k = tid * hper + i;
    if (k >= H) break;
    int v = cursor + k;
    if (v >= H) v -= H;
    my_free += !((in_use[v >> 5] >> (v & 31)) & 1u);
  }
  int total_free;
  int r = block_exclusive_scan(my_free, &total_free, s_warp);
  if (r < m) {
    for (int i = 0; i < hper; ++i) {
      const int k = tid * hper + i;
      if (k >= H || r >= m) break;
      int v = cursor + k;
      if (v >= H) v -= H;
      if (!((in_use[v >> 5] >> (v & 31)) & 1u)) victim[r++] = v;
    }
  }
  __syncthreads();
  const int mm = m < total_free ? m : total_free;  // misses that get a row

  // ---- read the previous owners (all reads before any write)
  int32_t evict[kMaxTokPerThread];
  r = miss_base;
#pragma unroll
  for (int i = 0; i < kMaxTokPerThread; ++i) {
    evict[i] = -1;
    if (tok[i] < 0) continue;
    if (r < mm) {
      const int v = victim[r];
      const int32_t e = owner[v];
      if (e >= 0 && (int64_t)e < n && (int64_t)slots[e] == hb + v) evict[i] = e;
    }
    ++r;
  }
  __syncthreads();

  // ---- writes: evicted owners go cold, misses take their rows; with
  // plan_only, each selected position also records the row its token is
  // copied into by the attention (-1: none)
  int2* fills = p.b.hot_fills + st * p.b.hot_fill_stride;
  int32_t* pend = p.b.hot_pend + st * p.b.hot_fill_stride;
  r = miss_base;
#pragma unroll
  for (int i = 0; i < kMaxTokPerThread; ++i) {
    const int j = tid * per + i;
    int32_t row = -1;
    if (tok[i] >= 0) {
      if (r < mm) {
        const int v = victim[r];
        if (evict[i] >= 0) slots[evict[i]] = -1;
        owner[v] = tok[i];
        row = (int32_t)(hb + v);
        slots[tok[i]] = row;
        fills[r] = make_int2(tok[i], row);
      }
      ++r;
    }
    if (p.plan_only && i < per && j < ntok) pend[j] = row;
  }
  if (tid == 0) {
    p.b.hot_nfill[st] = mm;
    p.b.hot_pend_on[st] = p.plan_only ? 1 : 0;
    if (mm > 0) p.b.hot_cursor[st] = victim[mm - 1] + 1 == H ? 0 : victim[mm - 1] + 1;
  }
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// kChunksPerRow: 16-byte chunks of a row (128 for BF16 rows, 65 for FP8 rows)
template <int kChunksPerRow>
__global__ void __launch_bounds__(kFillThreads) hot_fill_kernel(const HotParams p) {
  grid_dependency_wait();
  __shared__ const uint8_t* src[kFillRows];
  __shared__ uint8_t* dst[kFillRows];
  const int u = blockIdx.y;
  if (p.b.u[u].hot_base < 0 || p.b.hot_rows <= 0) return;
  const int64_t st = p.b.unit_state(u);
  const int nfill = p.b.hot_nfill[st];
  const int r0 = blockIdx.x * kFillRows;
  if (r0 >= nfill) return;
  if (threadIdx.x < kFillRows) {
    const int r = r0 + threadIdx.x;
    const uint8_t* sp = nullptr;
    uint8_t* dp = nullptr;
    if (r < nfill) {
      const int2 f = p.b.hot_fills[st * p.b.hot_fill_stride + r];
      const uint8_t* host = p.b.u[u].host_rows;
      if (host != nullptr && f.x >= 0 && (int64_t)f.x < p.b.u[u].n && f.y >= 0 &&
          (int64_t)f.y < p.b.pool_rows) {
        sp = host + (int64_t)f.x * (kChunksPerRow * 16);
        dp = p.b.pool + (int64_t)f.y * (kChunksPerRow * 16);
      } else {
        report_error(p.b.err, QSA_ERR_BAD_SLOT, kKernHot, ((int64_t)u << 40) | (uint32_t)r);
      }
    }
    src[threadIdx.x] = sp;
    dst[threadIdx.x] = dp;
  }
  __syncthreads();
  constexpr int kTotal = kFillRows * kChunksPerRow;
  constexpr int kPer = (kTotal + kFillThreads - 1) / kFillThreads;   // 4 or 3
  uint4 v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int idx = k * kFillThreads + threadIdx.x;
    const uint8_t* s = idx < kTotal ? src[idx / kChunksPerRow] : nullptr;
    v[k] = s ? ld_nc_v4(s + (idx % kChunksPerRow) * 16) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int idx = k * kFillThreads + threadIdx.x;
    if (idx < kTotal && src[idx / kChunksPerRow])
      *reinterpret_cast<uint4*>(dst[idx / kChunksPerRow] + (idx % kChunksPerRow) * 16) = v[k];
  }
}

}  // namespace

cudaError_t launch_hot_fetch(const BatchDesc& b, const int32_t* sel_blocks, const int32_t* n_sel,
                             int32_t budget_tokens, bool copy_rows, cudaStream_t s) {
  if (b.n_units <= 0 || b.hot_rows <= 0) return cudaSuccess;
  HotParams p;
  p.b = b;
  p.sel = sel_blocks;
  p.n_sel = n_sel;
  p.k_max = budget_tokens / 4;
  p.plan_only = copy_rows ? 0 : 1;
  const int smem = ((b.hot_rows + 31) / 32) * 4 + budget_tokens * 4;   // <= kPlanSmemMax
  cudaError_t e = launch_kernel(hot_plan_kernel, dim3(b.n_units), dim3(kPlanThreads), smem, s, 0,
                                dim3(1), p);
  if (e != cudaSuccess || !copy_rows) return e;
  dim3 grid((budget_tokens + kFillRows - 1) / kFillRows, b.n_units);
  if (b.row_bytes == kRowBytesFp8)
    return launch_kernel(hot_fill_kernel<kRowBytesFp8 / 16>, grid, dim3(kFillThreads), 0, s, 0, dim3(1), p);
  return launch_kernel(hot_fill_kernel<kRowBytes / 16>, grid, dim3(kFillThreads), 0, s, 0, dim3(1), p);
}

}  // namespace qsa
