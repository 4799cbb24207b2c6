// Internal declarations shared by the kernels and the C-ABI layer of the
// QSA decode-step library.  Not part of the public interface (include/qsa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "qsa.h"

namespace qsa {

constexpr int kIndexHeads = QSA_INDEX_HEADS;  // 8
constexpr int kIndexDim = QSA_INDEX_DIM;      // 64
constexpr int kKvHeads = QSA_KV_HEADS;        // 4
constexpr int kHeadDim = QSA_HEAD_DIM;        // 128
constexpr int kQHeads = QSA_Q_HEADS;          // 16
constexpr int kGroup = kQHeads / kKvHeads;    // 4 query heads per KV head
constexpr int kRowBytes = QSA_ROW_BYTES;      // 2048: BF16 row
constexpr int kRowBytesFp8 = QSA_ROW_BYTES_FP8;  // 1040: FP8 row
constexpr int kMaxUnits = QSA_MAX_UNITS;

// Split-K partial slots of the workspace: one per this many selected C4
// blocks of the budget (32 tokens), which caps the CTAs (partials) the
// attention gives one unit.  The no-allocation attention splits its rows in
// pieces of the same 32 tokens.
constexpr int kAttnBlocksPerSplit = 8;
constexpr int kAttnTokensPerSplit = kAttnBlocksPerSplit * 4;
// One split-K partial: running max m[16] and sum l[16] (base-2 logits), then
// the unnormalised accumulator acc[16][128].
constexpr int kPartFloats = kQHeads + kQHeads + kQHeads * kHeadDim;  // 2080
// Bytes at the start of the workspace reserved for the device error word.
constexpr int64_t kErrBytes = 256;

// Device error word.  The first kernel that meets a bad input records its
// status; later ones keep the first record.
struct ErrorWord {
  int32_t status;
  int32_t kernel;
  int64_t detail;
};

enum KernelId : int32_t {
  kKernIndexScore = 1,
  kKernTopk = 2,
  kKernGather = 3,
  kKernAttn = 4,
  kKernSlotFill = 5,
  kKernSlotSet = 6,
  kKernAppend = 7,
  kKernHot = 8,
};

// One decode unit (request slot, layer) of a call.
struct UnitDesc {
  int32_t req;                // request slot index
  int32_t layer;              // QSA layer
  int64_t n;                  // cached tokens of the request
  const uint8_t* host_rows;   // device-usable address of host row 0 of this
                              // (request, layer), or nullptr
  int64_t hot_base;           // first hot row of this (request, layer), or -1
};

// Everything a kernel needs to find a unit's data.  Passed by value.
struct BatchDesc {
  int32_t n_units;
  int32_t n_layers;           // layers per request in the cache layout
  int64_t ctx_cap;            // ctx_capacity of the cache layout
  int64_t pool_rows;
  const uint8_t* index_keys;  // [req][layer][ctx_cap][64]
  const uint16_t* index_scales;
  int32_t* slot_table;        // [req][layer][ctx_cap]
  uint8_t* pool;              // [pool_rows][2048]
  ErrorWord* err;
  float* partials;            // [req][layer][splits_max][kPartFloats]
  int32_t* tickets;           // [req][layer][2]: work counter, finished CTAs
  int32_t splits_max;
  int32_t row_bytes;          // kRowBytes (BF16 rows) or kRowBytesFp8 (FP8 rows)
  // Hot-cache state per (request, layer) (workspace; null without hot rows)
  int32_t hot_rows;           // rows per (request, layer); 0: no hot cache
  int32_t hot_fill_stride;    // entries of a fill list (the config's budget_tokens)
  int2* hot_fills;            // [req][layer][hot_fill_stride] {token, pool row}
  int32_t* hot_nfill;         // [req][layer] entries in the fill list
  int32_t* hot_cursor;        // [req][layer] next row to hand out
  int32_t* hot_owner;         // [req][layer][hot_rows] token held by a row, or -1
  // Misses planned by qsa_hot_cache_plan and not yet copied: per selected
  // position the pool row the attention fills from host memory (-1: none),
  // and per (request, layer) whether the map is live.
  int32_t* hot_pend;          // [req][layer][hot_fill_stride]
  int32_t* hot_pend_on;       // [req][layer]
  UnitDesc u[kMaxUnits];

  __host__ __device__ int64_t unit_row(int u_) const {
    return ((int64_t)u[u_].req * n_layers + u[u_].layer) * ctx_cap;
  }
  __host__ __device__ int64_t unit_state(int u_) const {
    return (int64_t)u[u_].req * n_layers + u[u_].layer;
  }
};

__device__ __forceinline__ void report_error(ErrorWord* e, int32_t status, int32_t kernel,
                                             int64_t detail) {
  if (atomicCAS(&e->status, 0, status) == 0) {
    e->kernel = kernel;
    e->detail = detail;
  }
}

// Source address of the 2048-byte row of logical token t of unit u, read
// through the slot table: pool row when the slot is >= 0, else the host
// history.  Returns nullptr (and records the error) for an invalid slot.
__device__ __forceinline__ const uint8_t* row_source(const BatchDesc& b, int u, int64_t t,
                                                     int32_t kernel) {
  const int32_t slot = b.slot_table[b.unit_row(u) + t];
  if (slot >= 0 && (int64_t)slot < b.pool_rows) return b.pool + (int64_t)slot * b.row_bytes;
  if (slot == -1 && b.u[u].host_rows != nullptr) return b.u[u].host_rows + t * b.row_bytes;
  report_error(b.err, QSA_ERR_BAD_SLOT, kernel, ((int64_t)u << 40) | (t & 0xFFFFFFFFFFll));
  return nullptr;
}

// Programmatic dependent launch.  Every hot-path kernel of the library is
// launched with programmatic stream serialization (launch_kernel below), and
// calls grid_dependency_wait() before its first global-memory access (set-up
// that touches only shared or tensor memory and the parameters comes first);
// it returns once the kernel before it on the stream has completed and its
// memory operations are visible (at once when there is none): measured on
// the 8 x 262144-token step, 1.191 -> 1.175 ms.  The main kernels also trigger their dependents
// where their CTAs' main work ends (trigger_dependents below).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel on the stream start launching once every CTA of this
// one has passed this point (its grid_dependency_wait() still waits for this
// kernel's completion and memory).  Called where a CTA's main work ends:
// the dependent's launch then overlaps this kernel's tail.  Measured on the
// HBM-resident chain (score, top-k, attention, merge per layer, one unit):
// 39.5 -> 37.5 us per layer; the two-micro-batch 256K step is unchanged
// (1.176 -> 1.172 ms).  A trigger at kernel start was slower everywhere (the
// chain 42.0 us per layer, the 256K step 1.239 against 1.215 ms, the 12-unit
// HBM attention 26 against 20 us): dependents held SMs while they waited.
// QSA_PDL_TRIGGER=0 removes the trigger.
#ifndef QSA_PDL_TRIGGER
#define QSA_PDL_TRIGGER 1
#endif
__device__ __forceinline__ void trigger_dependents() {
#if QSA_PDL_TRIGGER
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Launch `kernel` on stream s with programmatic stream serialization, an
// optional launch priority (0: the stream's) and optional cluster dims.
template <class... KArgs, class... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, int priority, dim3 cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (priority != 0) {
    attr[na].id = cudaLaunchAttributePriority;
    attr[na].val.priority = priority;
    ++na;
  }
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster.x;
    attr[na].val.clusterDim.y = cluster.y;
    attr[na].val.clusterDim.z = cluster.z;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Device ids the library keeps per-device state for.
constexpr int kMaxDevices = 64;

// One-time setup per device.  Kernel attributes set with cudaFuncSetAttribute
// apply to the device current on the calling thread, so every launcher runs
// its setup once for each device it launches on; the mutex serialises the
// first calls of concurrent threads.
class PerDeviceOnce {
 public:
  template <class F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices]{};
};

// SM count of the device current on the calling thread (queried once per
// device).
cudaError_t current_sm_count(int* out);

// Makes `dev` the calling thread's current device for the lifetime of the
// guard and restores the previous one afterwards (dev < 0: no change).
class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    if (dev < 0) return;
    status_ = cudaGetDevice(&prev_);
    if (status_ == cudaSuccess && prev_ != dev) {
      status_ = cudaSetDevice(dev);
      switched_ = status_ == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (switched_) cudaSetDevice(prev_);
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
  cudaError_t status() const { return status_; }

 private:
  int prev_ = 0;
  bool switched_ = false;
  cudaError_t status_ = cudaSuccess;
};

// Whether [p, p + bytes) lies inside host memory from qsa_host_alloc mapped
// for `device` (such memory is used by the device at its host address).
bool host_alloc_covers(const void* p, int64_t bytes, int device);

// Highest launch priority of the device (numerically lowest), for the
// attention launches: their CTAs are dispatched ahead of queued scoring CTAs
// of other requests.
int highest_priority();

// Record the thread-local message returned by qsa_last_error_string() and
// pass the status through (defined with the C ABI layer).
qsa_status_t set_last_error(qsa_status_t status, const char* message);

// Kernels of different calls share SMs (index score of some requests beside
// the attention of others on another stream).  An SM's split between L1 and
// shared memory is fixed while CTAs are resident on it, so every big kernel
// of the library asks for the largest shared-memory carveout: then a CTA
// never waits for an SM to drain just because another kernel chose a
// smaller split.
template <class Kernel>
cudaError_t prefer_max_shared(Kernel kernel, int dynamic_smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       dynamic_smem_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

// ------------------------------------------------------------ launchers
// Each returns the launch status (cudaGetLastError right after the launch).

// keys_map, scales_map: TMA tensor maps of the index keys (uint8 [rows][64])
// and scales (fp16 [rows]), rows = max_requests * n_layers * ctx_capacity
// (made by make_index_maps).
cudaError_t launch_index_score(const BatchDesc& b, const CUtensorMap* keys_map,
                               const CUtensorMap* scales_map, const float* q_idx, const float* w,
                               float* blk_scores, int64_t blk_stride, cudaStream_t s);

// Encode the tensor maps of the index keys at `keys` and the scales at
// `scales`, `rows` rows each.
cudaError_t make_index_maps(CUtensorMap* keys_map, const void* keys, CUtensorMap* scales_map,
                            const void* scales, int64_t rows);

cudaError_t launch_select_topk(const BatchDesc& b, const float* blk_scores, int64_t blk_stride,
                               int32_t k_max, int32_t* sel_blocks, int32_t* n_sel,
                               cudaStream_t s);

cudaError_t launch_gather_rows(const BatchDesc& b, const int32_t* sel_blocks,
                               const int32_t* n_sel, int32_t budget_tokens, uint8_t* rows_out,
                               int32_t* n_rows, cudaStream_t s);

cudaError_t launch_sparse_attn(const BatchDesc& b, const uint16_t* q, const int32_t* sel_blocks,
                               const int32_t* n_sel, int32_t budget_tokens,
                               const uint8_t* gathered, float softmax_scale, float* out,
                               float* lse, cudaStream_t s);

// Producer side: where each unit's newest token goes (computed from the
// leases on the host).  pool_row: the pool row that receives the row and
// becomes the token's slot (-1: none, the token is cold); evict: a token
// whose slot becomes -1 (a ring row handed to the new token), or -1.
struct AppendTargets {
  int64_t pool_row[kMaxUnits];
  int64_t evict[kMaxUnits];
};

cudaError_t launch_append_token(const BatchDesc& b, const AppendTargets& tg, const float* k_new,
                                const uint8_t* kv_new, cudaStream_t s);

// Cross-step hot cache: plan (slot, owner and cursor updates, fill lists)
// then the copy of the listed host rows into their hot rows.
// copy_rows = false: plan only; the next attention of the units reads the
// misses from host memory and writes them into their hot rows.
cudaError_t launch_hot_fetch(const BatchDesc& b, const int32_t* sel_blocks, const int32_t* n_sel,
                             int32_t budget_tokens, bool copy_rows, cudaStream_t s);

// Slot-table maintenance.
cudaError_t launch_slot_fill(int32_t* rows, int32_t n_layers, int64_t ctx_cap, int64_t ctx_len,
                             int32_t placement, int64_t row_base, int32_t layer_rows,
                             cudaStream_t s);

cudaError_t launch_slot_set(int32_t* row, int64_t ctx_len, int64_t pool_rows,
                            const int64_t* tokens, const int32_t* slots, int32_t n,
                            ErrorWord* err, cudaStream_t s);

}  // namespace qsa
