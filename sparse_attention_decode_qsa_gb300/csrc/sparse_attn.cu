// Step 4 of the QSA decode step: GQA decode attention over the selected
// rows only ("Оффлоадинг KV-кэша Qwen3.8-Flash-Next в RAM через vLLM без
// потери скорости декодирования", section "Механизм гибридного разреженного
// оффлоадинга": attention reads only the <= indexer_budget selected rows).
//
// Split-K flash-decode.  A split is 8 selected C4 blocks, i.e. 32 token
// rows (64 KiB of K/V).  Rows are read through the slot table (pool rows from
// HBM, cold rows zero-copy from mapped pinned host memory) or from a dense
// gathered buffer.
//
// Work layout: `cpu` CTAs per unit; CTA (unit u, slot r) takes the splits
// r, r + cpu, r + 2*cpu, ... of unit u and visits them alternately from the
// front and the back of that list.  Selected blocks are in ascending id order,
// so for a request with an HBM tail ring its early splits are cold (host) and
// its late splits hot (HBM): the alternation overlaps one split's host
// transfer with another split's compute.  Rows of the next split are copied
// with cp.async into the second of two 64 KiB buffers while the current
// split is computed.  A CTA keeps a running (max, sum, acc) across its splits
// (online softmax) and writes one partial; a small second kernel merges the
// cpu partials of each (unit, head) with the log-sum-exp rule.  When some
// row comes from host memory the grid is capped at kMaxCtasHost CTAs: that
// many SMs saturate the host link, and the rest stay free for HBM-bound work
// of other requests on other streams.
//
// Per split (256 threads):
//   logits : warp w serves KV head w/2 and 16 tokens; lane l holds dims
//            4l..4l+3 of the 4 query heads of that KV head, and the four
//            partial dots are reduced across the warp with a transposing
//            butterfly (6 shuffles for 4 values);
//   softmax: warp w owns query heads 2w, 2w+1, lane = token;
//   P.V    : thread t serves KV head t/64 and dims 2(t%64), 2(t%64)+1 of its
//            4 query heads.
// The products are plain FMAs: 4 query heads per KV head make this a
// 4-row contraction, not a tensor-core shape.
#include <cuda_bf16.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kSplitTokens = kAttnTokensPerSplit;     // 32
constexpr int kChunksPerRow = kRowBytes / 16;         // 128
constexpr int kBufBytes = kSplitTokens * kRowBytes;   // 64 KiB
constexpr int kSmemBytes = 2 * kBufBytes;             // double buffer
#ifndef QSA_ATTN_HOST_CTAS
#define QSA_ATTN_HOST_CTAS 64
#endif
constexpr int kMaxCtasHost = QSA_ATTN_HOST_CTAS;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  BatchDesc b;
  const uint16_t* q;        // [units][16][128] bf16 bits
  const int32_t* sel;       // [units][k_max]
  const int32_t* n_sel;
  int32_t k_max;
  int32_t budget_tokens;
  int32_t cpu;              // CTAs (partials) per unit
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
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// The k-th split this CTA visits (0 <= k < count): alternately from the front
// and the back of its list r, r + cpu, ...
__device__ __forceinline__ int visit_split(int k, int count, int r, int cpu) {
  const int idx = (k & 1) ? count - 1 - (k >> 1) : (k >> 1);
  return r + idx * cpu;
}

// Issue the copies of split `split` of unit u into buf; warp w copies rows
// 4w..4w+3, each lane 4 chunks of each.  valid[t] tells compute which rows
// exist (written by warp 0).
__device__ __forceinline__ void issue_split(const AttnParams& p, int u, int split, int nsel,
                                            uint8_t* buf, uint8_t* valid) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j0 = split * kAttnBlocksPerSplit;
  const int64_t n = p.b.u[u].n;
  // lane l resolves row l of the split (every warp does, so no block barrier)
  const uint8_t* src = nullptr;
  {
    const int j = j0 + lane / 4;
    if (j < nsel) {
      const int64_t b = p.sel[(int64_t)u * p.k_max + j];
      const int64_t t = 4 * b + (lane & 3);
      if (b < 0 || 4 * b >= n) {
        if ((lane & 3) == 0 && warp == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernAttn, b);
      } else if (t < n) {
        src = p.gathered ? p.gathered + ((int64_t)u * p.budget_tokens + 4 * j + (lane & 3)) * kRowBytes
                         : row_source(p.b, u, t, kKernAttn);
      }
    }
  }
  if (warp == 0) valid[lane] = src != nullptr;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = 4 * warp + r;
    const uint8_t* s = reinterpret_cast<const uint8_t*>(
        __shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(src), row));
#pragma unroll
    for (int c = 0; c < kChunksPerRow / 32; ++c) {
      const int chunk = c * 32 + lane;
      cp_async16(buf + row * kRowBytes + chunk * 16, s ? s + chunk * 16 : p.b.pool, s ? 16u : 0u);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_split_kernel(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t rows[];  // [2][32][2048]
  __shared__ uint8_t valid[2][kSplitTokens];
  __shared__ float logit[kQHeads][kSplitTokens];
  __shared__ float m_s[kQHeads], l_s[kQHeads];

  const int u = blockIdx.x / p.cpu, r = blockIdx.x % p.cpu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int nsel = p.n_sel[u];
  if (nsel < 0 || nsel > p.k_max) {
    if (r == 0 && tid == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernAttn, nsel);
    nsel = 0;
  }
  const int splits = (nsel + kAttnBlocksPerSplit - 1) / kAttnBlocksPerSplit;
  const int count = r < splits ? (splits - 1 - r) / p.cpu + 1 : 0;

  // query of this unit: warp w (KV head g = w/2) needs dims 4*lane.. of its 4 heads
  const int g_l = warp >> 1;
  float qr[kGroup][4];
  {
    const uint16_t* qu = p.q + (int64_t)u * kQHeads * kHeadDim;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const uint2 w2 = *reinterpret_cast<const uint2*>(qu + (g_l * kGroup + j) * kHeadDim + 4 * lane);
      qr[j][0] = bf16_lo(w2.x) * p.scale_log2;
      qr[j][1] = bf16_hi(w2.x) * p.scale_log2;
      qr[j][2] = bf16_lo(w2.y) * p.scale_log2;
      qr[j][3] = bf16_hi(w2.y) * p.scale_log2;
    }
  }
  // running state of this thread's P.V outputs: KV head g_v, dims d0, d0+1 of 4 heads
  const int g_v = tid >> 6, d0 = 2 * (tid & 63);
  float M[kGroup], L[kGroup], acc[kGroup][2];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) { M[j] = -INFINITY; L[j] = 0.f; acc[j][0] = acc[j][1] = 0.f; }

  int buf = 0;
  if (count > 0) issue_split(p, u, visit_split(0, count, r, p.cpu), nsel, rows, valid[0]);
  cp_async_commit();
  for (int k = 0; k < count; ++k) {
    if (k + 1 < count)
      issue_split(p, u, visit_split(k + 1, count, r, p.cpu), nsel, rows + (buf ^ 1) * kBufBytes,
                  valid[buf ^ 1]);
    cp_async_commit();
    cp_async_wait_1();  // this split's rows have landed (the next split's may still fly)
    __syncthreads();
    const uint8_t* R = rows + buf * kBufBytes;
    const uint8_t* V = valid[buf];

    // ---- logits (base 2): warp -> (KV head g_l, 16 tokens), lane -> 4 dims
    {
      const int tok0 = (warp & 1) * 16;
      const int hsel = (lane >> 3) & 3;  // head this lane ends up holding
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int tok = tok0 + i;
        const uint2 kk = *reinterpret_cast<const uint2*>(R + tok * kRowBytes + g_l * kHeadDim * 2 + lane * 8);
        const float k0 = bf16_lo(kk.x), k1 = bf16_hi(kk.x), k2 = bf16_lo(kk.y), k3 = bf16_hi(kk.y);
        float d[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j)
          d[j] = fmaf(qr[j][3], k3, fmaf(qr[j][2], k2, fmaf(qr[j][1], k1, qr[j][0] * k0)));
        // transposing butterfly: after it, lane l holds the full dot of head (l>>3)&3
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
        if ((lane & 7) == 0) logit[g_l * kGroup + hsel][tok] = V[tok] ? v : -INFINITY;
      }
    }
    __syncthreads();

    // ---- softmax within the split: warp -> heads 2w, 2w+1, lane -> token
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

    // ---- P.V and online-softmax update of the running state
    {
      float a[kGroup][2];
#pragma unroll
      for (int j = 0; j < kGroup; ++j) a[j][0] = a[j][1] = 0.f;
#pragma unroll 8
      for (int tok = 0; tok < kSplitTokens; ++tok) {
        const uint32_t vv = *reinterpret_cast<const uint32_t*>(
            R + tok * kRowBytes + kKvHeads * kHeadDim * 2 + g_v * kHeadDim * 2 + d0 * 2);
        const float v0 = bf16_lo(vv), v1 = bf16_hi(vv);
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          const float pr = logit[g_v * kGroup + j][tok];
          a[j][0] = fmaf(pr, v0, a[j][0]);
          a[j][1] = fmaf(pr, v1, a[j][1]);
        }
      }
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const float ms = m_s[g_v * kGroup + j];
        if (ms == -INFINITY) continue;                 // no token of this split
        const float mn = fmaxf(M[j], ms);
        const float so = exp2f(M[j] - mn), sn = exp2f(ms - mn);
        L[j] = fmaf(L[j], so, l_s[g_v * kGroup + j] * sn);
        acc[j][0] = fmaf(acc[j][0], so, a[j][0] * sn);
        acc[j][1] = fmaf(acc[j][1], so, a[j][1] * sn);
        M[j] = mn;
      }
    }
    __syncthreads();    // logit/m_s/l_s and this buffer are reused
    buf ^= 1;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");

  float* part = partial_ptr(p.b, u, r);
#pragma unroll
  for (int j = 0; j < kGroup; ++j)
    *reinterpret_cast<float2*>(part + 2 * kQHeads + (g_v * kGroup + j) * kHeadDim + d0) =
        make_float2(acc[j][0], acc[j][1]);
  if ((tid & 63) == 0) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      part[g_v * kGroup + j] = M[j];
      part[kQHeads + g_v * kGroup + j] = L[j];
    }
  }
}

// Merge: CTA (head, unit), thread = output dim; reads the cpu partials.
__global__ void __launch_bounds__(kHeadDim) attn_merge_kernel(const AttnParams p) {
  const int h = blockIdx.x, u = blockIdx.y, d = threadIdx.x;
  float Mx = -INFINITY;
  for (int s = 0; s < p.cpu; ++s) Mx = fmaxf(Mx, partial_ptr(p.b, u, s)[h]);
  float Lt = 0.f, acc = 0.f;
  if (Mx != -INFINITY) {
#pragma unroll 4
    for (int s = 0; s < p.cpu; ++s) {
      const float* part = partial_ptr(p.b, u, s);
      const float ms = part[h], ls = part[kQHeads + h], as = part[2 * kQHeads + h * kHeadDim + d];
      const float wgt = ms == -INFINITY ? 0.f : exp2f(ms - Mx);
      Lt = fmaf(wgt, ls, Lt);
      acc = fmaf(wgt, as, acc);
    }
  }
  float* o = p.out + ((int64_t)u * kQHeads + h) * kHeadDim;
  o[d] = Lt > 0.f ? acc / Lt : 0.f;
  if (p.lse && d == 0)
    p.lse[(int64_t)u * kQHeads + h] = Lt > 0.f ? (Mx + log2f(Lt)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_sparse_attn(const BatchDesc& b, const uint16_t* q, const int32_t* sel_blocks,
                               const int32_t* n_sel, int32_t budget_tokens,
                               const uint8_t* gathered, float softmax_scale, float* out,
                               float* lse, cudaStream_t s) {
  static bool attr_set = false;
  static int sm_count = 0;
  if (!attr_set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
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
  bool any_host = false;
  if (gathered == nullptr)
    for (int u = 0; u < b.n_units; ++u) any_host |= b.u[u].host_rows != nullptr;
  const int splits = (p.k_max + kAttnBlocksPerSplit - 1) / kAttnBlocksPerSplit;
  const int cap = any_host ? kMaxCtasHost : sm_count;
  int cpu = cap / b.n_units;
  if (cpu < 1) cpu = 1;
  if (cpu > splits) cpu = splits;
  p.cpu = cpu;
  attn_split_kernel<<<b.n_units * cpu, kThreads, kSmemBytes, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_merge_kernel<<<dim3(kQHeads, b.n_units), kHeadDim, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
