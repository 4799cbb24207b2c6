// Producer side of the QSA decode step: store the newest token of a unit.
// The token's index key is quantised to the compact 66-byte form the indexer
// reads (64 FP8-e4m3 codes + one fp16 scale: "Оффлоадинг KV-кэша
// Qwen3.8-Flash-Next в RAM через vLLM без потери скорости декодирования",
// section "Эффективность и память"), and its 2048-byte KV row goes where the
// request's placement keeps rows ("双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测",
// section "显存账本：热缓存卸载省下约84%": full history in pinned host memory,
// the newest tokens in an HBM tail ring, logical tokens kept apart from
// physical slots).
//
// One CTA of 128 threads per unit.  Threads 0-63 hold the 64 key elements:
// absmax by warp shuffles, scale = fp16 round-to-nearest-even of absmax/448
// (fp32 division, saturating at 65504), codes = E4M3 round-to-nearest-even
// (saturating) of clamp(k/scale, +-448) (fp32 division).  The row goes to
// the pool row and/or the host history row (a store through the mapped
// pointer crosses the host link): a BF16 row unchanged, 16 bytes per thread;
// for an FP8 cache each thread quantises 8 of the row's 1024 values under
// the same rule, one scale per 128-value head vector (16 threads each).
// Thread 0 writes the token's slot and, when a ring row is handed over,
// marks the token that held it cold.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 128;
static_assert(kRowBytes == kThreads * 16, "one 16-byte piece of the row per thread");
static_assert(kIndexDim == 64, "two warps hold the key");

struct AppendParams {
  BatchDesc b;
  AppendTargets tg;
  const float* k_new;       // [units][64]
  const uint8_t* kv_new;    // [units][2048]
};

__global__ void __launch_bounds__(kThreads) append_token_kernel(const AppendParams p) {
  grid_dependency_wait();
  __shared__ float s_amax[2];
  const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int64_t n = p.b.u[u].n;
  if (n < 1) {
    if (tid == 0) report_error(p.b.err, QSA_ERR_BAD_SLOT, kKernAppend, u);
    return;
  }
  const int64_t t = n - 1;
  const int64_t row = p.b.unit_row(u) + t;

  // ---- index key: absmax, fp16 scale, e4m3 codes
  float k = 0.f;
  if (tid < kIndexDim) k = p.k_new[(int64_t)u * kIndexDim + tid];
  float a = fabsf(k);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if (lane == 0 && tid < kIndexDim) s_amax[tid >> 5] = a;
  __syncthreads();
  const float amax = fmaxf(s_amax[0], s_amax[1]);
  const __half s16 = __float2half_rn(fminf(amax / 448.0f, 65504.0f));
  const float sf = __half2float(s16);
  if (tid < kIndexDim) {
    uint8_t code = 0;
    if (sf > 0.f) {
      const float x = fminf(fmaxf(k / sf, -448.0f), 448.0f);
      code = (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    }
    const_cast<uint8_t*>(p.b.index_keys)[row * kIndexDim + tid] = code;
  }
  if (tid == 0)
    const_cast<uint16_t*>(p.b.index_scales)[row] = sf > 0.f ? __half_as_ushort(s16) : (uint16_t)0;

  // ---- KV row
  const uint4 v = reinterpret_cast<const uint4*>(p.kv_new + (int64_t)u * kRowBytes)[tid];
  const int64_t pool_row = p.tg.pool_row[u];
  const bool to_pool = pool_row >= 0 && pool_row < p.b.pool_rows;
  if (pool_row >= p.b.pool_rows && tid == 0) report_error(p.b.err, QSA_ERR_BAD_SLOT, kKernAppend, pool_row);
  uint8_t* dst_pool = to_pool ? p.b.pool + pool_row * p.b.row_bytes : nullptr;
  uint8_t* dst_host = p.b.u[u].host_rows ? const_cast<uint8_t*>(p.b.u[u].host_rows) + t * p.b.row_bytes
                                         : nullptr;
  if (p.b.row_bytes == kRowBytes) {
    if (dst_pool) reinterpret_cast<uint4*>(dst_pool)[tid] = v;
    if (dst_host) reinterpret_cast<uint4*>(dst_host)[tid] = v;
  } else {
    // head vector hv = tid / 16 (K heads 0-3, then V heads 0-3), values
    // 8 (tid % 16) .. +7 of it; the BF16 row holds them in this order
    float x[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float va = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) va = fmaxf(va, fabsf(x[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) va = fmaxf(va, __shfl_xor_sync(0xFFFFFFFFu, va, o));
    const __half vs16 = __float2half_rn(fminf(va / 448.0f, 65504.0f));
    const float vsf = __half2float(vs16);
    uint32_t packed[2] = {0u, 0u};
    if (vsf > 0.f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float y = fminf(fmaxf(x[i] / vsf, -448.0f), 448.0f);
        packed[i >> 2] |= (uint32_t)(uint8_t)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3)
                          << (8 * (i & 3));
      }
    }
    const uint2 codes = make_uint2(packed[0], packed[1]);
    const int hv = tid >> 4;
    const int off = hv * kHeadDim + (tid & 15) * 8;          // K codes, then V codes
    const uint16_t sbits = vsf > 0.f ? __half_as_ushort(vs16) : (uint16_t)0;
    if (dst_pool) {
      *reinterpret_cast<uint2*>(dst_pool + off) = codes;
      if ((tid & 15) == 0) reinterpret_cast<uint16_t*>(dst_pool + 2 * kKvHeads * kHeadDim)[hv] = sbits;
    }
    if (dst_host) {
      *reinterpret_cast<uint2*>(dst_host + off) = codes;
      if ((tid & 15) == 0) reinterpret_cast<uint16_t*>(dst_host + 2 * kKvHeads * kHeadDim)[hv] = sbits;
    }
  }

  // ---- slot table
  if (tid == 0) {
    int32_t* slots = p.b.slot_table + p.b.unit_row(u);
    slots[t] = to_pool ? (int32_t)pool_row : -1;
    const int64_t ev = p.tg.evict[u];
    if (ev >= 0 && ev < t) slots[ev] = -1;
  }
}

}  // namespace

cudaError_t launch_append_token(const BatchDesc& b, const AppendTargets& tg, const float* k_new,
                                const uint8_t* kv_new, cudaStream_t s) {
  if (b.n_units <= 0) return cudaSuccess;
  AppendParams p;
  p.b = b;
  p.tg = tg;
  p.k_new = k_new;
  p.kv_new = kv_new;
  return launch_kernel(append_token_kernel, dim3(b.n_units), dim3(kThreads), 0, s, 0, dim3(1), p);
}

}  // namespace qsa
