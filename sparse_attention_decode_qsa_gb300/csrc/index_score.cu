// Step 1 of the QSA decode step: the resident indexer.  Every cached token t
// of a unit is scored from its compact key (64 FP8-e4m3 codes + one fp16
// scale, 66 bytes):
//     S_t = sum_h w_h * relu(scale_t * sum_d q[h][d] * e4m3(code_t[d]))
// and the scores are reduced to C4 blocks (max over 4 adjacent tokens) in the
// same pass, so only one fp32 per block leaves the kernel.
// Sources: "Оффлоадинг KV-кэша Qwen3.8-Flash-Next в RAM через vLLM без потери
// скорости декодирования", section "Механизм гибридного разреженного
// оффлоадинга" (resident indexer over 66-byte keys), and
// "双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测", opening explanation of
// QSA (C4 blocks of 4 adjacent tokens).
//
// Mapping: one thread owns one C4 block (4 tokens, 256 bytes of codes), so
// every query value read from shared memory feeds four tokens' FMAs.  The
// query is kept transposed in shared memory ([dim][head]) so one pair of
// 16-byte loads gives all 8 heads of one dimension.  Tiles of 512 tokens from
// all units of the call form one flat grid.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

#ifdef QSA_INDEX_SCORE_FFMA
constexpr int kThreads = 128;              // one C4 block per thread
constexpr int kTileTokens = kThreads * 4;  // 512
#endif

struct IndexScoreParams {
  BatchDesc b;
  int32_t tile_start[kMaxUnits + 1];  // prefix sums of tiles per unit
  const float* q_idx;                 // [units][8][64]
  const float* w;                     // [units][8]
  float* blk;                         // [units][blk_stride]
  int64_t blk_stride;
};

#ifdef QSA_INDEX_SCORE_FFMA
// CUDA-core version (fp32 FMAs), kept for A/B comparison builds.
__device__ __forceinline__ uint4 ldg_stream(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Two e4m3 codes (low byte first) to two floats, via the hardware
// e4m3x2 -> f16x2 conversion (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair16) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)pair16, __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

__global__ void __launch_bounds__(kThreads) index_score_kernel(const IndexScoreParams p) {
  __shared__ __align__(16) float qs[kIndexDim][kIndexHeads];
  __shared__ float ws[kIndexHeads];

  const int tile = blockIdx.x;
  int lo = 0, hi = p.b.n_units - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int u = lo;

  const float* qu = p.q_idx + (int64_t)u * kIndexHeads * kIndexDim;
  for (int i = threadIdx.x; i < kIndexHeads * kIndexDim; i += kThreads)
    qs[i % kIndexDim][i / kIndexDim] = qu[i];
  if (threadIdx.x < kIndexHeads) ws[threadIdx.x] = p.w[(int64_t)u * kIndexHeads + threadIdx.x];
  __syncthreads();

  const int64_t n = p.b.u[u].n;
  const int64_t blk = (int64_t)(tile - p.tile_start[u]) * kThreads + threadIdx.x;
  const int64_t t0 = blk * 4;
  if (t0 >= n) return;
  const int nt = (n - t0) < 4 ? (int)(n - t0) : 4;
  const int64_t row = p.b.unit_row(u) + t0;
  const uint8_t* kp = p.b.index_keys + row * kIndexDim;
  const uint16_t* sp = p.b.index_scales + row;

  float acc[4][kIndexHeads];
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int h = 0; h < kIndexHeads; ++h) acc[t][h] = 0.f;

#pragma unroll
  for (int c = 0; c < 4; ++c) {  // 16-dim chunks of the 64 dims
    uint4 kv[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      kv[t] = (t < nt) ? ldg_stream(kp + t * kIndexDim + c * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // dim pairs within the chunk
      const int d = c * 16 + 2 * j;
      const float4 qa0 = *reinterpret_cast<const float4*>(&qs[d][0]);
      const float4 qa1 = *reinterpret_cast<const float4*>(&qs[d][4]);
      const float4 qb0 = *reinterpret_cast<const float4*>(&qs[d + 1][0]);
      const float4 qb1 = *reinterpret_cast<const float4*>(&qs[d + 1][4]);
      const float qa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
      const float qb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t word = (j >> 1) == 0 ? kv[t].x : (j >> 1) == 1 ? kv[t].y
                            : (j >> 1) == 2 ? kv[t].z : kv[t].w;
        const float2 kf = e4m3x2_to_float2((j & 1) ? (word >> 16) : (word & 0xFFFFu));
#pragma unroll
        for (int h = 0; h < kIndexHeads; ++h) {
          acc[t][h] = fmaf(kf.x, qa[h], acc[t][h]);
          acc[t][h] = fmaf(kf.y, qb[h], acc[t][h]);
        }
      }
    }
  }

  float best = -INFINITY;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    if (t < nt) {
      const float sc = __half2float(__ushort_as_half(sp[t]));
      float s = 0.f;
#pragma unroll
      for (int h = 0; h < kIndexHeads; ++h) s = fmaf(ws[h], fmaxf(acc[t][h] * sc, 0.f), s);
      best = fmaxf(best, s);
    }
  }
  p.blk[(int64_t)u * p.blk_stride + blk] = best;
}


#endif  // QSA_INDEX_SCORE_FFMA

// ---------------------------------------------------------------------------
// Tensor-core version (tcgen05, 5th-generation tensor cores with TMEM
// accumulators).  The scan does 512 multiply-adds per 66 bytes, more than the
// CUDA cores deliver at HBM speed, and it is a genuine dense contraction:
// keys[tokens][64] x q^T[64][8 heads].
//
// Per CTA: 8 tiles of M = 128 tokens.  A tile's codes are converted exactly
// to f16 (every e4m3 value is an f16 value) and stored as the A operand; the
// B operand holds the index query split as q = hi + lo (both f16, hi = f16(q),
// lo = f16(q - hi)), so N = 16 columns: 8 heads x {hi, lo}, which keeps the
// product at fp32 accuracy.  Four tcgen05.mma (K = 16 each) accumulate the
// fp32 dots of a tile in 16 TMEM columns; two such column blocks alternate
// between tiles, so the epilogue of tile i-1 (tcgen05.ld, relu, head weights,
// scale, C4 max through shuffles) runs while the MMAs of tile i execute and
// the codes of tile i+1 are being loaded.  Thread t owns token t of a tile in
// every phase: it loads and converts that token's row, and TMEM lane t holds
// its accumulators.
//
// Operand layout: K-major without swizzle, made of core matrices of 8 rows x
// 16 bytes (8 f16).  Element (row, k) of a K-step of 16 lies at
// (row/8)*256 + ((k%16)/8)*128 + (row%8)*16 + (k%8)*2 bytes; the descriptor's
// leading byte offset (next core matrix along K) is 128 and its stride byte
// offset (next 8-row group) is 256.
constexpr int kTcThreads = 128;
constexpr int kTcTile = 128;
constexpr int kTcTilesPerCta = 8;
constexpr int kTcCtaTokens = kTcTile * kTcTilesPerCta;  // 1024
constexpr uint32_t kTmemCols = 32;                     // two 16-column accumulators
constexpr int kAStageBytes = kTcTile * kIndexDim * 2;  // 16 KiB
constexpr int kAKStepBytes = kTcTile * 16 * 2;         // 4 KiB
constexpr int kBBytes = 16 * kIndexDim * 2;            // 2 KiB
constexpr int kBKStepBytes = 16 * 16 * 2;              // 512 B
constexpr int kTcSmemBytes = 2 * kAStageBytes + kBBytes + 64;
// kind::f16 instruction descriptor: D f32 (bit 4), A = B = f16, both K-major,
// N/8 at bits 17-22, M/16 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kWaitPolls = 1u << 20;              // bounded mbarrier waits

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return (uint32_t)__cvta_generic_to_shared(ptr);
}

__device__ __forceinline__ uint32_t kmajor_off(int row, int k, int kstep_bytes) {
  return (k >> 4) * kstep_bytes + (row >> 3) * 256 + ((k >> 3) & 1) * 128 + (row & 7) * 16 +
         (k & 7) * 2;
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (all >> 4), descriptor version 1 at bit 46, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint4 ld_keys(const uint8_t* ptr) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair16) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)pair16, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

__global__ void __launch_bounds__(kTcThreads) index_score_tc_kernel(const IndexScoreParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sA = smem;                                         // [2][16 KiB]
  uint8_t* sB = smem + 2 * kAStageBytes;                      // 2 KiB
  uint64_t* bar = reinterpret_cast<uint64_t*>(sB + kBBytes);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int lo = 0, hi = p.b.n_units - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.tile_start[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
  }
  const int u = lo;
  const int64_t n = p.b.u[u].n;
  const int64_t t_cta = (int64_t)(blockIdx.x - p.tile_start[u]) * kTcCtaTokens;
  const int64_t left = n - t_cta;
  const int n_tiles = (int)((left + kTcTile - 1) / kTcTile < kTcTilesPerCta
                                ? (left + kTcTile - 1) / kTcTile : kTcTilesPerCta);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)), "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // B operand: rows 0..7 = f16(q_h), rows 8..15 = f16(q_h - f16(q_h))
  {
    const float* qu = p.q_idx + (int64_t)u * kIndexHeads * kIndexDim;
    for (int i = tid; i < kIndexHeads * kIndexDim; i += kTcThreads) {
      const int h = i >> 6, d = i & 63;
      const float qv = qu[i];
      const __half qh = __float2half_rn(qv);
      const __half ql = __float2half_rn(qv - __half2float(qh));
      *reinterpret_cast<__half*>(sB + kmajor_off(h, d, kBKStepBytes)) = qh;
      *reinterpret_cast<__half*>(sB + kmajor_off(h + 8, d, kBKStepBytes)) = ql;
    }
  }
  float w[kIndexHeads];
#pragma unroll
  for (int h = 0; h < kIndexHeads; ++h) w[h] = p.w[(int64_t)u * kIndexHeads + h];
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t row0 = p.b.unit_row(u);
  const uint8_t* keys = p.b.index_keys + row0 * kIndexDim;
  const uint16_t* scl = p.b.index_scales + row0;
  float* out = p.blk + (int64_t)u * p.blk_stride;
  const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);

  uint4 raw[4];
  {
    const int64_t t = t_cta + tid;
#pragma unroll
    for (int c = 0; c < 4; ++c) raw[c] = t < n ? ld_keys(keys + t * kIndexDim + c * 16) : make_uint4(0, 0, 0, 0);
  }
  float sc_prev = 0.f;
  bool ok = true;

  // epilogue of tile j: accumulators -> score -> C4 max -> block score
  auto epilogue = [&](int j, float sc) {
    const int b = j & 1;
    uint32_t polls = 0;
    while (!mbar_try_wait(&bar[b], (uint32_t)(j >> 1) & 1u)) {
      if (++polls > kWaitPolls) {
        report_error(p.b.err, QSA_ERR_TIMEOUT, kKernIndexScore, j);
        ok = false;
        break;
      }
    }
    tc_fence_after();
    float v[16];
    tc_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * 16), v);
    const int64_t tok = t_cta + (int64_t)j * kTcTile + tid;
    float s = -INFINITY;
    if (tok < n) {
      s = 0.f;
#pragma unroll
      for (int h = 0; h < kIndexHeads; ++h) s = fmaf(w[h], fmaxf((v[h] + v[h + 8]) * sc, 0.f), s);
    }
    s = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
    s = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
    if ((lane & 3) == 0 && tok < n) out[tok >> 2] = s;
  };

  int done = 0;
  for (int i = 0; i < n_tiles; ++i) {
    if (!__syncthreads_and(ok)) break;
    const int b = i & 1;
    uint4 cur[4] = {raw[0], raw[1], raw[2], raw[3]};
    const int64_t tok = t_cta + (int64_t)i * kTcTile + tid;
    const float sc_cur = tok < n ? __half2float(__ushort_as_half(scl[tok])) : 0.f;
    if (i + 1 < n_tiles) {
      const int64_t t = tok + kTcTile;
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[c] = t < n ? ld_keys(keys + t * kIndexDim + c * 16) : make_uint4(0, 0, 0, 0);
    }
    // convert this thread's token row into A[b]
    uint8_t* a = sA + b * kAStageBytes + (tid >> 3) * 256 + (tid & 7) * 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t wd[4] = {cur[c].x, cur[c].y, cur[c].z, cur[c].w};
      uint32_t h[8];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        h[2 * m] = e4m3x2_to_f16x2(wd[m] & 0xFFFFu);
        h[2 * m + 1] = e4m3x2_to_f16x2(wd[m] >> 16);
      }
      *reinterpret_cast<uint4*>(a + c * kAKStepBytes) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(a + c * kAKStepBytes + 128) = make_uint4(h[4], h[5], h[6], h[7]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t d = tmem + (uint32_t)(b * 16);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc_mma_f16(d, smem_desc(a_base + b * kAStageBytes + k * kAKStepBytes, 128, 256),
                   smem_desc(b_base + k * kBKStepBytes, 128, 256), k > 0 ? 1u : 0u);
      tc_commit(&bar[b]);
    }
    if (i >= 1) epilogue(i - 1, sc_prev);
    sc_prev = sc_cur;
    done = i + 1;
  }
  if (__syncthreads_and(ok) && done > 0) epilogue(done - 1, sc_prev);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
}
}  // namespace

cudaError_t launch_index_score(const BatchDesc& b, const float* q_idx, const float* w,
                               float* blk_scores, int64_t blk_stride, cudaStream_t s) {
#ifdef QSA_INDEX_SCORE_FFMA
  const int cta_tokens = kTileTokens;
#else
  const int cta_tokens = kTcCtaTokens;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(index_score_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
#endif
  IndexScoreParams p;
  p.b = b;
  p.q_idx = q_idx;
  p.w = w;
  p.blk = blk_scores;
  p.blk_stride = blk_stride;
  int64_t tiles = 0;
  for (int u = 0; u < b.n_units; ++u) {
    p.tile_start[u] = (int32_t)tiles;
    tiles += (b.u[u].n + cta_tokens - 1) / cta_tokens;
  }
  p.tile_start[b.n_units] = (int32_t)tiles;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
#ifdef QSA_INDEX_SCORE_FFMA
  index_score_kernel<<<(unsigned)tiles, kThreads, 0, s>>>(p);
#else
  index_score_tc_kernel<<<(unsigned)tiles, kTcThreads, kTcSmemBytes, s>>>(p);
#endif
  return cudaGetLastError();
}

}  // namespace qsa
