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

constexpr int kThreads = 128;              // one C4 block per thread
constexpr int kTileTokens = kThreads * 4;  // 512

struct IndexScoreParams {
  BatchDesc b;
  int32_t tile_start[kMaxUnits + 1];  // prefix sums of tiles per unit
  const float* q_idx;                 // [units][8][64]
  const float* w;                     // [units][8]
  float* blk;                         // [units][blk_stride]
  int64_t blk_stride;
};

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

}  // namespace

cudaError_t launch_index_score(const BatchDesc& b, const float* q_idx, const float* w,
                               float* blk_scores, int64_t blk_stride, cudaStream_t s) {
  IndexScoreParams p;
  p.b = b;
  p.q_idx = q_idx;
  p.w = w;
  p.blk = blk_scores;
  p.blk_stride = blk_stride;
  int64_t tiles = 0;
  for (int u = 0; u < b.n_units; ++u) {
    p.tile_start[u] = (int32_t)tiles;
    tiles += (b.u[u].n + kTileTokens - 1) / kTileTokens;
  }
  p.tile_start[b.n_units] = (int32_t)tiles;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  index_score_kernel<<<(unsigned)tiles, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
