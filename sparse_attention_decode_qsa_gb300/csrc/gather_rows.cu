// Step 3 of the QSA decode step and the slot-table maintenance kernels.
//
// The slot table keeps logical token addresses apart from physical cache
// slots; selected rows are found through it, in the HBM pool (tail ring,
// staging or resident rows) or, for cold tokens, in the request's pinned host
// history, and only those rows are moved ("双卡RTX4090跑通Qwen3-Next：8并发满血
// 长上下文实测", section "显存账本：热缓存卸载省下约84%"; "Оффлоадинг KV-кэша
// Qwen3.8-Flash-Next в RAM через vLLM без потери скорости декодирования",
// section "Механизм гибридного разреженного оффлоадинга").
//
// Gather mapping: a CTA owns 8 selected blocks (32 token rows: 64 KiB of BF16
// rows, 32.5 KiB of FP8 rows).  Its first warp resolves the 32 row sources
// into shared memory; then all 256 threads copy 16-byte chunks (16 each for
// BF16 rows, 9 for FP8 rows), all loads issued before the stores so that
// many requests are in flight on the host link.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherBlocks = 8;
constexpr int kGatherRows = kGatherBlocks * 4;

struct GatherParams {
  BatchDesc b;
  const int32_t* sel;
  const int32_t* n_sel;
  int32_t k_max;
  int32_t budget_tokens;
  uint8_t* out;      // [units][budget_tokens][row bytes]
  int32_t* n_rows;   // [units] or nullptr
};

__device__ __forceinline__ uint4 ld_nc_v4(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// kChunksPerRow: 16-byte chunks of a row (128 for BF16 rows, 65 for FP8 rows)
template <int kChunksPerRow>
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const GatherParams p) {
  grid_dependency_wait();
  __shared__ const uint8_t* src[kGatherRows];
  const int u = blockIdx.y;
  const int j0 = blockIdx.x * kGatherBlocks;
  const int64_t n = p.b.u[u].n;
  int nsel = p.n_sel[u];
  if (nsel < 0 || nsel > p.k_max) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernGather, nsel);
    return;
  }
  if (threadIdx.x == 0 && blockIdx.x == 0 && p.n_rows != nullptr) {
    int32_t rows = 0;
    if (nsel > 0) {
      const int64_t blast = p.sel[(int64_t)u * p.k_max + nsel - 1];
      const int64_t last = n - 4 * blast;
      rows = 4 * (nsel - 1) + (int32_t)(last < 0 ? 0 : (last > 4 ? 4 : last));
    }
    p.n_rows[u] = rows;
  }
  if (j0 >= nsel) return;

  if (threadIdx.x < kGatherRows) {
    const int j = j0 + threadIdx.x / 4;
    const uint8_t* ptr = nullptr;
    if (j < nsel) {
      const int64_t b = p.sel[(int64_t)u * p.k_max + j];
      const int64_t t = 4 * b + (threadIdx.x & 3);
      if (b < 0 || 4 * b >= n) {
        if ((threadIdx.x & 3) == 0) report_error(p.b.err, QSA_ERR_BAD_BLOCK, kKernGather, b);
      } else if (t < n) {
        ptr = row_source(p.b, u, t, kKernGather);
      }
    }
    src[threadIdx.x] = ptr;
  }
  __syncthreads();

  uint8_t* dst = p.out + ((int64_t)u * p.budget_tokens + 4 * (int64_t)j0) * (kChunksPerRow * 16);
  constexpr int kTotal = kGatherRows * kChunksPerRow;
  constexpr int kPer = (kTotal + kGatherThreads - 1) / kGatherThreads;  // 16 or 9
  uint4 v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int idx = k * kGatherThreads + threadIdx.x;
    const uint8_t* s = idx < kTotal ? src[idx / kChunksPerRow] : nullptr;
    v[k] = s ? ld_nc_v4(s + (idx % kChunksPerRow) * 16) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int idx = k * kGatherThreads + threadIdx.x;
    if (idx < kTotal && src[idx / kChunksPerRow])
      *reinterpret_cast<uint4*>(dst + (int64_t)idx * 16) = v[k];
  }
}

// Fill the slot-table rows of a new request (all layers).
__global__ void slot_fill_kernel(int32_t* rows, int32_t n_layers, int64_t ctx_cap, int64_t ctx_len,
                                 int32_t placement, int64_t row_base, int32_t layer_rows) {
  const int64_t total = (int64_t)n_layers * ctx_len;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t l = i / ctx_len, t = i % ctx_len;
    int64_t slot;
    if (placement == QSA_KV_HBM) {
      slot = row_base + l * layer_rows + t;
    } else if (placement == QSA_KV_HOST) {
      slot = -1;
    } else {
      slot = (t >= ctx_len - layer_rows) ? row_base + l * layer_rows + (t % layer_rows) : -1;
    }
    rows[l * ctx_cap + t] = (int32_t)slot;
  }
}

__global__ void slot_set_kernel(int32_t* row, int64_t ctx_len, int64_t pool_rows,
                                const int64_t* tokens, const int32_t* slots, int32_t n,
                                ErrorWord* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t t = tokens[i];
  const int32_t s = slots[i];
  if (t < 0 || t >= ctx_len || s < -1 || (int64_t)s >= pool_rows) {
    report_error(err, QSA_ERR_BAD_SLOT, kKernSlotSet, i);
    return;
  }
  row[t] = s;
}

}  // namespace

cudaError_t launch_gather_rows(const BatchDesc& b, const int32_t* sel_blocks,
                               const int32_t* n_sel, int32_t budget_tokens, uint8_t* rows_out,
                               int32_t* n_rows, cudaStream_t s) {
  GatherParams p;
  p.b = b;
  p.sel = sel_blocks;
  p.n_sel = n_sel;
  p.k_max = budget_tokens / 4;
  p.budget_tokens = budget_tokens;
  p.out = rows_out;
  p.n_rows = n_rows;
  static PerDeviceOnce setup;
  cudaError_t e0 = setup.run([] {
    cudaError_t e = cudaFuncSetAttribute(gather_rows_kernel<kRowBytes / 16>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gather_rows_kernel<kRowBytesFp8 / 16>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    return e;
  });
  if (e0 != cudaSuccess) return e0;
  dim3 grid((p.k_max + kGatherBlocks - 1) / kGatherBlocks, b.n_units);
  if (b.row_bytes == kRowBytesFp8)
    return launch_kernel(gather_rows_kernel<kRowBytesFp8 / 16>, grid, dim3(kGatherThreads), 0, s, 0,
                         dim3(1), p);
  return launch_kernel(gather_rows_kernel<kRowBytes / 16>, grid, dim3(kGatherThreads), 0, s, 0, dim3(1), p);
}

cudaError_t launch_slot_fill(int32_t* rows, int32_t n_layers, int64_t ctx_cap, int64_t ctx_len,
                             int32_t placement, int64_t row_base, int32_t layer_rows,
                             cudaStream_t s) {
  const int64_t total = (int64_t)n_layers * ctx_len;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) return cudaSuccess;
  slot_fill_kernel<<<(unsigned)blocks, threads, 0, s>>>(rows, n_layers, ctx_cap, ctx_len,
                                                        placement, row_base, layer_rows);
  return cudaGetLastError();
}

cudaError_t launch_slot_set(int32_t* row, int64_t ctx_len, int64_t pool_rows,
                            const int64_t* tokens, const int32_t* slots, int32_t n,
                            ErrorWord* err, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  slot_set_kernel<<<(n + 255) / 256, 256, 0, s>>>(row, ctx_len, pool_rows, tokens, slots, n, err);
  return cudaGetLastError();
}

}  // namespace qsa
