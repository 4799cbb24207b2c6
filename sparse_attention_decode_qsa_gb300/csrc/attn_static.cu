// Decode attention over a dense buffer of gathered KV rows, with its split-K
// scratch in a fixed device array of this library instead of caller memory.
//
// For callers that cannot allocate device memory at the point where they run
// attention: code inside a serving engine whose device memory is handed out
// by a pre-planned arena it may not grow, plug-ins that get only the buffers
// of their inputs and outputs, and code paths where calling cudaMalloc would
// synchronise the device or is forbidden.  They pass the query, the rows and
// the outputs; the split-K partials live in g_attn_scratch below.
//
// It computes what qsa_sparse_decode_attn computes from gathered rows, but
// with its own work layout: one CTA per 32 gathered rows, where the main
// kernel's CTAs stream 16-row splits and keep a running softmax state.  The
// two sum and merge in a different order, so they agree to rounding (far
// inside the 2e-3 attention tolerance).
#include <cuda_runtime.h>

#include <mutex>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kSplitTokens = kAttnTokensPerSplit;  // 32 rows per CTA
constexpr int kChunksPerRow = kRowBytes / 16;
constexpr int kSmemBytes = kSplitTokens * kRowBytes;
constexpr int kStaticSplits = QSA_STATIC_MAX_ROWS / kSplitTokens;  // 64
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One (m[16], l[16], acc[16][128]) partial per (unit, split): 8.5 MB.  Every
// GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) float
    g_attn_scratch[QSA_STATIC_MAX_UNITS * kStaticSplits * kPartFloats];

struct StaticAttnParams {
  const uint16_t* q;      // [units][16][128] bf16 bits
  const uint8_t* rows;    // [units][rows_stride][2048]
  const int32_t* n_rows;  // [units]
  int32_t rows_stride;
  float scale_log2;
  float* out;             // [units][16][128]
  float* lse;             // [units][16] or nullptr
  float* scratch;         // device address of g_attn_scratch
};

__device__ __forceinline__ int valid_rows(const StaticAttnParams& p, int u) {
  const int n = p.n_rows[u];
  return n < 0 ? 0 : (n > p.rows_stride ? p.rows_stride : n);
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads) static_attn_split(const StaticAttnParams p) {
  extern __shared__ __align__(16) uint8_t rows[];
  __shared__ float logit[kQHeads][kSplitTokens];
  __shared__ float m_s[kQHeads], l_s[kQHeads];
  const int u = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = valid_rows(p, u);
  const int r0 = split * kSplitTokens;
  if (r0 >= n) return;
  const int nr = (n - r0) < kSplitTokens ? (n - r0) : kSplitTokens;
  const uint8_t* src = p.rows + ((int64_t)u * p.rows_stride + r0) * kRowBytes;
  {
    constexpr int kPer = kSplitTokens * kChunksPerRow / kThreads;
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int idx = k * kThreads + tid;
      v[k] = (idx / kChunksPerRow < nr)
                 ? __ldg(reinterpret_cast<const uint4*>(src + (int64_t)idx * 16))
                 : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      *reinterpret_cast<uint4*>(rows + (k * kThreads + tid) * 16) = v[k];
  }
  __syncthreads();
  {
    const int g = warp >> 1, tok0 = (warp & 1) * 16;
    float qr[kGroup][4];
    const uint16_t* qu = p.q + (int64_t)u * kQHeads * kHeadDim;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const uint2 w2 = *reinterpret_cast<const uint2*>(qu + (g * kGroup + j) * kHeadDim + 4 * lane);
      qr[j][0] = bf16_lo(w2.x) * p.scale_log2;
      qr[j][1] = bf16_hi(w2.x) * p.scale_log2;
      qr[j][2] = bf16_lo(w2.y) * p.scale_log2;
      qr[j][3] = bf16_hi(w2.y) * p.scale_log2;
    }
    const int hsel = (lane >> 3) & 3;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      const uint2 kk = *reinterpret_cast<const uint2*>(rows + tok * kRowBytes + g * kHeadDim * 2 + lane * 8);
      const float k0 = bf16_lo(kk.x), k1 = bf16_hi(kk.x), k2 = bf16_lo(kk.y), k3 = bf16_hi(kk.y);
      float d[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j)
        d[j] = fmaf(qr[j][3], k3, fmaf(qr[j][2], k2, fmaf(qr[j][1], k1, qr[j][0] * k0)));
      const bool up16 = lane & 16;
      const float a0 = up16 ? d[0] : d[2], a1 = up16 ? d[1] : d[3];
      const float r0v = __shfl_xor_sync(0xFFFFFFFFu, a0, 16);
      const float r1v = __shfl_xor_sync(0xFFFFFFFFu, a1, 16);
      const float v0 = (up16 ? d[2] : d[0]) + r0v;
      const float v1 = (up16 ? d[3] : d[1]) + r1v;
      const bool up8 = lane & 8;
      const float a = up8 ? v0 : v1;
      float v = (up8 ? v1 : v0) + __shfl_xor_sync(0xFFFFFFFFu, a, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
      if ((lane & 7) == 0) logit[g * kGroup + hsel][tok] = tok < nr ? v : -INFINITY;
    }
  }
  __syncthreads();
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = 2 * warp + hh;
    const float x = logit[h][lane];
    float m = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float pr = (x == -INFINITY) ? 0.f : exp2f(x - m);
    float l = pr;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    logit[h][lane] = pr;
    if (lane == 0) { m_s[h] = m; l_s[h] = l; }
  }
  __syncthreads();
  float* part = p.scratch + ((int64_t)u * kStaticSplits + split) * kPartFloats;
  {
    const int g = tid >> 6, d0 = 2 * (tid & 63);
    float acc[kGroup][2];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) acc[j][0] = acc[j][1] = 0.f;
#pragma unroll 8
    for (int tok = 0; tok < kSplitTokens; ++tok) {
      const uint32_t vv = *reinterpret_cast<const uint32_t*>(
          rows + tok * kRowBytes + kKvHeads * kHeadDim * 2 + g * kHeadDim * 2 + d0 * 2);
      const float v0 = bf16_lo(vv), v1 = bf16_hi(vv);
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const float pr = logit[g * kGroup + j][tok];
        acc[j][0] = fmaf(pr, v0, acc[j][0]);
        acc[j][1] = fmaf(pr, v1, acc[j][1]);
      }
    }
#pragma unroll
    for (int j = 0; j < kGroup; ++j)
      *reinterpret_cast<float2*>(part + 2 * kQHeads + (g * kGroup + j) * kHeadDim + d0) =
          make_float2(acc[j][0], acc[j][1]);
  }
  if (tid < kQHeads) {
    part[tid] = m_s[tid];
    part[kQHeads + tid] = l_s[tid];
  }
}

__global__ void __launch_bounds__(kHeadDim) static_attn_merge(const StaticAttnParams p) {
  const int h = blockIdx.x, u = blockIdx.y, d = threadIdx.x;
  const int n = valid_rows(p, u);
  float* o = p.out + ((int64_t)u * kQHeads + h) * kHeadDim;
  const int splits = (n + kSplitTokens - 1) / kSplitTokens;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s)
    M = fmaxf(M, p.scratch[((int64_t)u * kStaticSplits + s) * kPartFloats + h]);
  float L = 0.f, acc = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float* part = p.scratch + ((int64_t)u * kStaticSplits + s) * kPartFloats;
      const float ms = part[h];
      if (ms == -INFINITY) continue;
      const float wgt = exp2f(ms - M);
      L = fmaf(wgt, part[kQHeads + h], L);
      acc = fmaf(wgt, part[2 * kQHeads + h * kHeadDim + d], acc);
    }
  }
  o[d] = L > 0.f ? acc / L : 0.f;
  if (p.lse && d == 0)
    p.lse[(int64_t)u * kQHeads + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

// Device address of g_attn_scratch per device, looked up once per device.
std::mutex g_setup_mutex;
float* g_scratch_addr[kMaxDevices] = {};
bool g_smem_set[kMaxDevices] = {};

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" qsa_status_t qsa_sparse_decode_attn_noalloc(const uint16_t* q, const void* rows,
                                                       const int32_t* n_rows, int32_t n_units,
                                                       int32_t rows_stride, float softmax_scale,
                                                       float* out, float* lse, void* stream) {
  if (!q || !rows || !n_rows || !out) return set_last_error(QSA_ERR_INVALID_ARG, "null array");
  if (n_units < 1 || n_units > QSA_STATIC_MAX_UNITS)
    return set_last_error(QSA_ERR_INVALID_ARG,
                          "n_units must be in [1, QSA_STATIC_MAX_UNITS = 16]; split the batch");
  if (rows_stride < 1 || rows_stride > QSA_STATIC_MAX_ROWS)
    return set_last_error(QSA_ERR_INVALID_ARG,
                          "rows_stride must be in [1, QSA_STATIC_MAX_ROWS = 2048]");
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(rows) % 16)
    return set_last_error(QSA_ERR_INVALID_ARG, "q and rows must be 16-byte aligned");
  if (!(softmax_scale == softmax_scale))
    return set_last_error(QSA_ERR_INVALID_ARG, "softmax_scale is NaN");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_last_error(QSA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_last_error(QSA_ERR_INVALID_ARG, "device id too large");
  float* scratch;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_attn_scratch);
      if (e != cudaSuccess) return set_last_error(QSA_ERR_CUDA, cudaGetErrorString(e));
      g_scratch_addr[dev] = static_cast<float*>(ptr);
    }
    if (!g_smem_set[dev]) {
      e = cudaFuncSetAttribute(static_attn_split, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
      if (e != cudaSuccess) return set_last_error(QSA_ERR_CUDA, cudaGetErrorString(e));
      g_smem_set[dev] = true;
    }
    scratch = g_scratch_addr[dev];
  }
  StaticAttnParams p;
  p.q = q;
  p.rows = static_cast<const uint8_t*>(rows);
  p.n_rows = n_rows;
  p.rows_stride = rows_stride;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = out;
  p.lse = lse;
  p.scratch = scratch;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int splits = (rows_stride + kSplitTokens - 1) / kSplitTokens;
  static_attn_split<<<dim3(splits, n_units), kThreads, kSmemBytes, s>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    static_attn_merge<<<dim3(kQHeads, n_units), kHeadDim, 0, s>>>(p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return set_last_error(QSA_ERR_CUDA, cudaGetErrorString(e));
  return set_last_error(QSA_OK, "");
}
