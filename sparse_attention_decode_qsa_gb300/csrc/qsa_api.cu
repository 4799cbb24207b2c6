// C ABI of the QSA decode-step library and its host-side cache manager.
//
// The cache manager follows "双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测",
// section "显存账本：热缓存卸载省下约84%": the full KV history of a long
// request stays in pinned host memory, the GPU keeps a hot tail ring per
// request plus a shared staging area, logical token addresses are kept apart
// from physical cache slots (the slot table), and requests hold leases with
// generation tags so that a finished or cancelled request gives its capacity
// and slots back and a new request can reuse them safely.
//
// Host state: one lease per request slot and a first-fit free list of HBM
// pool row ranges.  Device state (all caller-allocated): the pool, the index
// keys, the slot table and the workspace (error word, split-K partials, and
// the index-score work counters of every request x layer).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <map>
#include <new>
#include <string>
#include <vector>

#include "qsa_internal.cuh"

using namespace qsa;

namespace {

thread_local std::string g_last_error;

qsa_status_t fail(qsa_status_t st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
qsa_status_t fail(qsa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

qsa_status_t ok() {
  g_last_error.clear();
  return QSA_OK;
}

qsa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(QSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct Lease {
  uint32_t generation = 0;
  bool active = false;
  int64_t ctx_len = 0;
  int64_t max_ctx = 0;                 // row stride of the HBM region / host history
  int32_t placement = 0;
  int32_t layer_rows = 0;
  int64_t row_base = 0;
  int64_t rows = 0;
  int64_t hot_base = -1;               // first hot row, or -1
  const uint8_t* host_rows = nullptr;  // device-usable address
};

int64_t splits_max_of(const qsa_cache_config& c) {
  const int64_t kmax = c.budget_tokens / 4;
  return (kmax + kAttnBlocksPerSplit - 1) / kAttnBlocksPerSplit;
}

bool config_sizes_ok(const qsa_cache_config* c) {
  return c && c->n_layers > 0 && c->max_requests > 0 && c->ctx_capacity > 0 &&
         c->ctx_capacity <= 0x7FFFFFFFll && c->budget_tokens >= 4 &&
         c->budget_tokens % 4 == 0 && c->budget_tokens <= QSA_MAX_BUDGET_TOKENS &&
         c->ring_tokens > 0 && c->staging_rows >= 0 && c->hbm_pool_rows >= 0 &&
         c->hbm_pool_rows <= 0x7FFFFFFFll && (c->kv_format == QSA_KV_BF16 || c->kv_format == QSA_KV_FP8) &&
         (c->hot_rows == 0 || (c->hot_rows >= c->budget_tokens && c->hot_rows <= QSA_MAX_HOT_ROWS)) &&
         c->reserved1 == 0;
}

// Workspace layout: error word, split-K partials, index-score work counters,
// then (hot_rows > 0) the hot-cache state.  Byte offsets.
struct WorkspaceLayout {
  int64_t partials, tickets, hot_fills, hot_nfill, hot_cursor, hot_owner, hot_pend, hot_pend_on,
      total;
};

WorkspaceLayout workspace_layout(const qsa_cache_config& c) {
  const int64_t units = (int64_t)c.max_requests * c.n_layers;
  WorkspaceLayout w;
  w.partials = kErrBytes;
  w.tickets = w.partials + units * splits_max_of(c) * kPartFloats * (int64_t)sizeof(float);
  w.hot_fills = w.tickets + units * 2 * (int64_t)sizeof(int32_t);   // 8-byte aligned
  const bool hot = c.hot_rows > 0;
  w.hot_nfill = w.hot_fills + (hot ? units * c.budget_tokens * (int64_t)sizeof(int2) : 0);
  w.hot_cursor = w.hot_nfill + (hot ? units * (int64_t)sizeof(int32_t) : 0);
  w.hot_owner = w.hot_cursor + (hot ? units * (int64_t)sizeof(int32_t) : 0);
  w.hot_pend = w.hot_owner + (hot ? units * c.hot_rows * (int64_t)sizeof(int32_t) : 0);
  w.hot_pend_on = w.hot_pend + (hot ? units * c.budget_tokens * (int64_t)sizeof(int32_t) : 0);
  w.total = w.hot_pend_on + (hot ? units * (int64_t)sizeof(int32_t) : 0);
  return w;
}

}  // namespace

int qsa::highest_priority() {
  static const int prio = [] {   // thread-safe one-time initialisation
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) {
      cudaGetLastError();
      greatest = 0;
    }
    return greatest;
  }();
  return prio;
}

cudaError_t qsa::current_sm_count(int* out) {
  static std::atomic<int> counts[kMaxDevices];   // 0: not yet queried
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int v = counts[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    counts[dev].store(v, std::memory_order_relaxed);
  }
  *out = v;
  return cudaSuccess;
}


qsa_status_t qsa::set_last_error(qsa_status_t status, const char* message) {
  g_last_error = message ? message : "";
  return status;
}

struct qsa_cache {
  CUtensorMap keys_map;       // TMA views of the index keys and scales (64-byte aligned)
  CUtensorMap scales_map;
  qsa_cache_config cfg;
  bool has_device = false;
  int device = -1;            // CUDA device of the device storage (-1: host-only cache)
  int64_t staging_total = 0;
  int64_t splits_max = 0;
  std::vector<Lease> leases;
  std::map<int64_t, int64_t> free_rows;  // start -> length

  ErrorWord* err() const { return reinterpret_cast<ErrorWord*>(cfg.workspace); }
  int64_t row_bytes() const { return cfg.kv_format == QSA_KV_FP8 ? kRowBytesFp8 : kRowBytes; }
  template <class T>
  T* ws_at(int64_t off) const {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(cfg.workspace) + off);
  }
  float* partials() const { return ws_at<float>(workspace_layout(cfg).partials); }
  int32_t* tickets() const { return ws_at<int32_t>(workspace_layout(cfg).tickets); }

  bool alloc_rows(int64_t n, int64_t* base) {
    for (auto it = free_rows.begin(); it != free_rows.end(); ++it) {
      if (it->second >= n) {
        *base = it->first;
        const int64_t rest = it->second - n, start = it->first + n;
        free_rows.erase(it);
        if (rest > 0) free_rows[start] = rest;
        return true;
      }
    }
    return false;
  }

  void release_rows(int64_t base, int64_t n) {
    if (n <= 0) return;
    auto next = free_rows.lower_bound(base);
    if (next != free_rows.end() && base + n == next->first) {
      n += next->second;
      next = free_rows.erase(next);
    }
    if (next != free_rows.begin()) {
      auto prev = std::prev(next);
      if (prev->first + prev->second == base) {
        prev->second += n;
        return;
      }
    }
    free_rows[base] = n;
  }

  // Every call that touches device storage runs on the cache's device (a
  // DeviceGuard makes it current) and refuses a stream of another device:
  // here when the stream is not being captured (a stream's device cannot be
  // queried during capture), else through the launch, which fails for a
  // stream that does not belong to the current device.
  qsa_status_t check_stream(void* stream, const DeviceGuard& g) const {
    if (device < 0) return QSA_OK;
    if (g.status() != cudaSuccess) return cuda_fail(g.status(), "making the cache's device current");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread) return QSA_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "querying the stream's capture status");
    if (cs != cudaStreamCaptureStatusNone) return QSA_OK;
    int sdev = -1;
    e = cudaStreamGetDevice(s, &sdev);
    if (e != cudaSuccess) return cuda_fail(e, "querying the stream's device");
    if (sdev != device)
      return fail(QSA_ERR_INVALID_ARG, "stream belongs to device %d, the cache's storage to device %d",
                  sdev, device);
    return QSA_OK;
  }

  qsa_status_t check_handle(qsa_handle h, const Lease** out) const {
    if (h.index >= leases.size())
      return fail(QSA_ERR_STALE_HANDLE, "request index %u out of range", h.index);
    const Lease& l = leases[h.index];
    if (!l.active || l.generation != h.generation)
      return fail(QSA_ERR_STALE_HANDLE, "stale handle {%u, %u} (live generation %u, %s)", h.index,
                  h.generation, l.generation, l.active ? "active" : "free");
    *out = &l;
    return QSA_OK;
  }

  // Validate a batch and describe its units for the kernels.
  qsa_status_t build_batch(const qsa_batch* b, BatchDesc* d) const {
    if (!has_device) return fail(QSA_ERR_NO_DEVICE, "cache has no device storage");
    if (!b || !b->requests) return fail(QSA_ERR_INVALID_ARG, "null batch");
    if (b->n_req <= 0 || b->n_layers <= 0 || b->layer0 < 0 ||
        (int64_t)b->layer0 + b->n_layers > cfg.n_layers)
      return fail(QSA_ERR_INVALID_ARG, "bad batch shape n_req=%d layer0=%d n_layers=%d",
                  b->n_req, b->layer0, b->n_layers);
    if ((int64_t)b->n_req * b->n_layers > kMaxUnits)
      return fail(QSA_ERR_INVALID_ARG, "batch has %lld units, limit %d",
                  (long long)b->n_req * b->n_layers, kMaxUnits);
    d->n_units = b->n_req * b->n_layers;
    d->n_layers = cfg.n_layers;
    d->ctx_cap = cfg.ctx_capacity;
    d->pool_rows = cfg.hbm_pool_rows;
    d->index_keys = cfg.index_keys;
    d->index_scales = cfg.index_scales;
    d->slot_table = cfg.slot_table;
    d->pool = static_cast<uint8_t*>(cfg.hbm_pool);
    d->err = err();
    d->partials = partials();
    d->tickets = tickets();
    d->splits_max = (int32_t)splits_max;
    d->row_bytes = (int32_t)row_bytes();
    const WorkspaceLayout w = workspace_layout(cfg);
    const bool hot = cfg.hot_rows > 0;
    d->hot_rows = cfg.hot_rows;
    d->hot_fill_stride = cfg.budget_tokens;
    d->hot_fills = hot ? ws_at<int2>(w.hot_fills) : nullptr;
    d->hot_nfill = hot ? ws_at<int32_t>(w.hot_nfill) : nullptr;
    d->hot_cursor = hot ? ws_at<int32_t>(w.hot_cursor) : nullptr;
    d->hot_owner = hot ? ws_at<int32_t>(w.hot_owner) : nullptr;
    d->hot_pend = hot ? ws_at<int32_t>(w.hot_pend) : nullptr;
    d->hot_pend_on = hot ? ws_at<int32_t>(w.hot_pend_on) : nullptr;
    for (int i = 0; i < b->n_req; ++i) {
      const Lease* l;
      if (qsa_status_t st = check_handle(b->requests[i], &l)) return st;
      for (int k = 0; k < i; ++k)
        if (b->requests[k].index == b->requests[i].index)
          return fail(QSA_ERR_INVALID_ARG, "request %u appears twice in the batch",
                      b->requests[i].index);
      for (int li = 0; li < b->n_layers; ++li) {
        UnitDesc& u = d->u[li * b->n_req + i];
        u.req = (int32_t)b->requests[i].index;
        u.layer = b->layer0 + li;
        u.n = l->ctx_len;
        u.host_rows = l->host_rows ? l->host_rows + (int64_t)u.layer * l->max_ctx * row_bytes()
                                   : nullptr;
        u.hot_base = l->hot_base >= 0 ? l->hot_base + (int64_t)u.layer * cfg.hot_rows : -1;
      }
    }
    return QSA_OK;
  }
};

extern "C" {

int32_t qsa_abi_version(void) { return QSA_ABI_VERSION; }

const char* qsa_last_error_string(void) { return g_last_error.c_str(); }

int64_t qsa_workspace_bytes(const qsa_cache_config* c) {
  if (!config_sizes_ok(c)) return -1;
  return workspace_layout(*c).total;
}

qsa_status_t qsa_cache_create(const qsa_cache_config* c, qsa_cache** out) {
  if (!out) return fail(QSA_ERR_INVALID_ARG, "null output pointer");
  *out = nullptr;
  if (!config_sizes_ok(c)) return fail(QSA_ERR_INVALID_ARG, "bad cache config sizes");
  const bool any = c->hbm_pool || c->index_keys || c->index_scales || c->slot_table || c->workspace;
  const bool all = c->hbm_pool && c->index_keys && c->index_scales && c->slot_table && c->workspace;
  if (any && !all)
    return fail(QSA_ERR_INVALID_ARG, "device storage must be given completely or not at all");
  if (all) {
    if (c->workspace_bytes < qsa_workspace_bytes(c))
      return fail(QSA_ERR_INVALID_ARG, "workspace has %lld bytes, needs %lld",
                  (long long)c->workspace_bytes, (long long)qsa_workspace_bytes(c));
    const void* ptrs[] = {c->hbm_pool, c->index_keys, c->index_scales, c->slot_table, c->workspace};
    for (const void* p : ptrs)
      if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
        return fail(QSA_ERR_INVALID_ARG, "device buffers must be 16-byte aligned");
  }
  int device = -1;
  if (all) {
    // the device storage must live on one device, which every call then uses
    const void* ptrs[] = {c->hbm_pool, c->index_keys, c->index_scales, c->slot_table, c->workspace};
    for (const void* p : ptrs) {
      cudaPointerAttributes a{};
      cudaError_t e = cudaPointerGetAttributes(&a, p);
      if (e != cudaSuccess) return cuda_fail(e, "querying a device buffer");
      if (a.type != cudaMemoryTypeDevice)
        return fail(QSA_ERR_INVALID_ARG, "device storage must be device memory");
      if (device >= 0 && a.device != device)
        return fail(QSA_ERR_INVALID_ARG, "device storage spans devices %d and %d", device, a.device);
      device = a.device;
    }
  }
  DeviceGuard guard(device);
  if (guard.status() != cudaSuccess) return cuda_fail(guard.status(), "making the storage's device current");
  const int64_t staging = (int64_t)c->n_layers * c->staging_rows;
  if (staging > c->hbm_pool_rows)
    return fail(QSA_ERR_CAPACITY, "staging (%lld rows) does not fit the pool (%lld rows)",
                (long long)staging, (long long)c->hbm_pool_rows);

  qsa_cache* cache = new (std::nothrow) qsa_cache();
  if (!cache) return fail(QSA_ERR_INVALID_ARG, "out of host memory");
  cache->cfg = *c;
  cache->has_device = all;
  cache->device = device;
  cache->staging_total = staging;
  cache->splits_max = splits_max_of(*c);
  cache->leases.resize(c->max_requests);
  if (c->hbm_pool_rows > staging) cache->free_rows[staging] = c->hbm_pool_rows - staging;

  if (all) {
    const int64_t key_rows = (int64_t)c->max_requests * c->n_layers * c->ctx_capacity;
    if (key_rows >= (1ll << 31)) {
      delete cache;
      return fail(QSA_ERR_INVALID_ARG, "%lld index-key rows exceed the 2^31 rows a TMA view addresses",
                  (long long)key_rows);
    }
    cudaError_t e = make_index_maps(&cache->keys_map, c->index_keys, &cache->scales_map,
                                    c->index_scales, key_rows);
    if (e != cudaSuccess) {
      delete cache;
      return cuda_fail(e, "encoding the index-key tensor maps");
    }
    e = cudaMemset(c->workspace, 0, (size_t)c->workspace_bytes);
    if (e == cudaSuccess)
      e = cudaMemset(c->slot_table, 0xFF,
                     (size_t)c->max_requests * c->n_layers * c->ctx_capacity * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      delete cache;
      return cuda_fail(e, "initialising workspace and slot table");
    }
  }
  *out = cache;
  return ok();
}

qsa_status_t qsa_cache_destroy(qsa_cache* cache) {
  delete cache;
  return ok();
}

qsa_status_t qsa_request_begin(qsa_cache* c, const qsa_request_desc* desc, void* stream,
                               qsa_handle* out) {
  if (!c || !desc || !out) return fail(QSA_ERR_INVALID_ARG, "null argument");
  if (desc->ctx_len < 1) return fail(QSA_ERR_INVALID_ARG, "ctx_len must be >= 1");
  if (desc->ctx_len > c->cfg.ctx_capacity)
    return fail(QSA_ERR_CAPACITY, "ctx_len %lld exceeds capacity %lld", (long long)desc->ctx_len,
                (long long)c->cfg.ctx_capacity);
  if (desc->max_ctx < 0 || desc->max_ctx > c->cfg.ctx_capacity)
    return fail(QSA_ERR_CAPACITY, "max_ctx %d outside [0, %lld]", desc->max_ctx,
                (long long)c->cfg.ctx_capacity);
  if (desc->max_ctx > 0 && desc->max_ctx < desc->ctx_len)
    return fail(QSA_ERR_INVALID_ARG, "max_ctx %d < ctx_len %lld", desc->max_ctx,
                (long long)desc->ctx_len);
  const int64_t max_ctx = desc->max_ctx > 0 ? desc->max_ctx : desc->ctx_len;
  if (desc->placement != QSA_KV_HBM && desc->placement != QSA_KV_HOST_RING &&
      desc->placement != QSA_KV_HOST)
    return fail(QSA_ERR_INVALID_ARG, "unknown placement %d", desc->placement);
  if (desc->placement != QSA_KV_HBM && !desc->host_rows)
    return fail(QSA_ERR_INVALID_ARG, "host placements need host_rows");
  if (desc->placement == QSA_KV_HBM && desc->host_rows)
    return fail(QSA_ERR_INVALID_ARG, "HBM placement takes no host_rows");

  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  int slot = -1;
  for (size_t i = 0; i < c->leases.size(); ++i)
    if (!c->leases[i].active) { slot = (int)i; break; }
  if (slot < 0) return fail(QSA_ERR_OUT_OF_SLOTS, "all %d request slots are leased", c->cfg.max_requests);

  const int32_t layer_rows = desc->placement == QSA_KV_HBM        ? (int32_t)max_ctx
                             : desc->placement == QSA_KV_HOST_RING ? c->cfg.ring_tokens
                                                                   : 0;
  const bool hot = desc->placement != QSA_KV_HBM && c->cfg.hot_rows > 0;
  const int64_t ring_rows = (int64_t)layer_rows * c->cfg.n_layers;
  const int64_t rows = ring_rows + (hot ? (int64_t)c->cfg.hot_rows * c->cfg.n_layers : 0);

  const uint8_t* host_dev = nullptr;
  if (desc->placement != QSA_KV_HBM) {
    if (c->has_device) {
      const int64_t need = (int64_t)c->cfg.n_layers * max_ctx * c->row_bytes();
      if (host_alloc_covers(desc->host_rows, need, c->device)) {
        host_dev = static_cast<const uint8_t*>(desc->host_rows);   // same address on the device
      } else {
        void* dptr = nullptr;
        cudaError_t e = cudaHostGetDevicePointer(&dptr, const_cast<void*>(desc->host_rows), 0);
        if (e != cudaSuccess) {
          cudaGetLastError();
          return fail(QSA_ERR_INVALID_ARG,
                      "host_rows is neither qsa_host_alloc memory nor pinned, mapped host memory: %s",
                      cudaGetErrorString(e));
        }
        host_dev = static_cast<const uint8_t*>(dptr);
      }
    } else {
      host_dev = static_cast<const uint8_t*>(desc->host_rows);
    }
    if (reinterpret_cast<uintptr_t>(host_dev) % 16 != 0)
      return fail(QSA_ERR_INVALID_ARG, "host_rows must be 16-byte aligned");
  }

  int64_t base = 0;
  if (rows > 0 && !c->alloc_rows(rows, &base))
    return fail(QSA_ERR_CAPACITY, "no free pool range of %lld rows", (long long)rows);

  if (c->has_device) {
    int32_t* st = c->cfg.slot_table + (int64_t)slot * c->cfg.n_layers * c->cfg.ctx_capacity;
    cudaError_t e = launch_slot_fill(st, c->cfg.n_layers, c->cfg.ctx_capacity, desc->ctx_len,
                                     desc->placement, base, layer_rows,
                                     static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess && hot) {
      // every hot row of the request free, cursors at row 0
      const WorkspaceLayout w = workspace_layout(c->cfg);
      const int64_t st0 = (int64_t)slot * c->cfg.n_layers;
      e = cudaMemsetAsync(c->ws_at<int32_t>(w.hot_owner) + st0 * c->cfg.hot_rows, 0xFF,
                          (size_t)c->cfg.n_layers * c->cfg.hot_rows * sizeof(int32_t),
                          static_cast<cudaStream_t>(stream));
      if (e == cudaSuccess)
        e = cudaMemsetAsync(c->ws_at<int32_t>(w.hot_cursor) + st0, 0,
                            (size_t)c->cfg.n_layers * sizeof(int32_t), static_cast<cudaStream_t>(stream));
      if (e == cudaSuccess)   // no planned rows pending a copy
        e = cudaMemsetAsync(c->ws_at<int32_t>(w.hot_pend_on) + st0, 0,
                            (size_t)c->cfg.n_layers * sizeof(int32_t), static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) {
      c->release_rows(base, rows);
      return cuda_fail(e, "slot-table fill");
    }
  }

  Lease& l = c->leases[slot];
  l.generation += 1;
  l.active = true;
  l.ctx_len = desc->ctx_len;
  l.max_ctx = max_ctx;
  l.placement = desc->placement;
  l.layer_rows = layer_rows;
  l.row_base = base;
  l.rows = rows;
  l.hot_base = hot ? base + ring_rows : -1;
  l.host_rows = host_dev;
  out->index = (uint32_t)slot;
  out->generation = l.generation;
  return ok();
}

qsa_status_t qsa_request_end(qsa_cache* c, qsa_handle h) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  const Lease* cl;
  if (qsa_status_t st = c->check_handle(h, &cl)) return st;
  Lease& l = c->leases[h.index];
  c->release_rows(l.row_base, l.rows);
  l.active = false;
  l.ctx_len = 0;
  l.max_ctx = 0;
  l.rows = 0;
  l.hot_base = -1;
  l.host_rows = nullptr;
  return ok();
}

qsa_status_t qsa_request_info_get(qsa_cache* c, qsa_handle h, qsa_request_info* out) {
  if (!c || !out) return fail(QSA_ERR_INVALID_ARG, "null argument");
  const Lease* l;
  if (qsa_status_t st = c->check_handle(h, &l)) return st;
  out->ctx_len = l->ctx_len;
  out->placement = l->placement;
  out->layer_rows = l->layer_rows;
  out->hbm_row_base = l->row_base;
  out->host_rows = l->host_rows;
  out->max_ctx = l->max_ctx;
  out->hot_row_base = l->hot_base;
  return ok();
}

qsa_status_t qsa_request_advance(qsa_cache* c, qsa_handle h, int32_t n_new) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  const Lease* cl;
  if (qsa_status_t st = c->check_handle(h, &cl)) return st;
  if (n_new < 1) return fail(QSA_ERR_INVALID_ARG, "n_new %d < 1", n_new);
  Lease& l = c->leases[h.index];
  if (l.ctx_len + n_new > l.max_ctx)
    return fail(QSA_ERR_CAPACITY, "ctx_len %lld + %d exceeds the request's max_ctx %lld",
                (long long)l.ctx_len, n_new, (long long)l.max_ctx);
  l.ctx_len += n_new;
  return ok();
}

qsa_status_t qsa_cache_stats(const qsa_cache* c, qsa_stats* out) {
  if (!c || !out) return fail(QSA_ERR_INVALID_ARG, "null argument");
  std::memset(out, 0, sizeof *out);
  out->max_requests = c->cfg.max_requests;
  int64_t leased = 0;
  for (const Lease& l : c->leases) {
    if (l.active) { out->active_requests++; leased += l.rows; }
  }
  out->free_request_slots = c->cfg.max_requests - out->active_requests;
  out->free_ranges = (int32_t)c->free_rows.size();
  out->hbm_pool_rows = c->cfg.hbm_pool_rows;
  for (const auto& kv : c->free_rows) {
    out->free_hbm_rows += kv.second;
    if (kv.second > out->largest_free_rows) out->largest_free_rows = kv.second;
  }
  out->staging_rows_total = c->staging_total;
  out->hbm_kv_bytes_in_use = leased * c->row_bytes();
  return ok();
}

qsa_status_t qsa_slot_table_ptr(qsa_cache* c, qsa_handle h, int32_t layer, int32_t** out) {
  if (!c || !out) return fail(QSA_ERR_INVALID_ARG, "null argument");
  if (!c->has_device) return fail(QSA_ERR_NO_DEVICE, "cache has no device storage");
  const Lease* l;
  if (qsa_status_t st = c->check_handle(h, &l)) return st;
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(QSA_ERR_INVALID_ARG, "bad layer %d", layer);
  *out = c->cfg.slot_table + ((int64_t)h.index * c->cfg.n_layers + layer) * c->cfg.ctx_capacity;
  return ok();
}

qsa_status_t qsa_slot_table_set(qsa_cache* c, qsa_handle h, int32_t layer, const int64_t* tokens,
                                const int32_t* slots, int32_t n, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  int32_t* row = nullptr;
  if (qsa_status_t st = qsa_slot_table_ptr(c, h, layer, &row)) return st;
  if (n < 0 || (n > 0 && (!tokens || !slots))) return fail(QSA_ERR_INVALID_ARG, "bad token/slot arrays");
  cudaError_t e = launch_slot_set(row, c->leases[h.index].ctx_len, c->cfg.hbm_pool_rows, tokens,
                                  slots, n, c->err(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "slot-table set");
  return ok();
}

qsa_status_t qsa_staging_ptr(qsa_cache* c, int32_t layer, void** out) {
  if (!c || !out) return fail(QSA_ERR_INVALID_ARG, "null argument");
  if (!c->has_device) return fail(QSA_ERR_NO_DEVICE, "cache has no device storage");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(QSA_ERR_INVALID_ARG, "bad layer %d", layer);
  *out = static_cast<uint8_t*>(c->cfg.hbm_pool) + (int64_t)layer * c->cfg.staging_rows * c->row_bytes();
  return ok();
}

qsa_status_t qsa_poll_error(qsa_cache* c, void* stream, int32_t* dev_status, int64_t* detail) {
  if (!c || !dev_status) return fail(QSA_ERR_INVALID_ARG, "null argument");
  if (!c->has_device) return fail(QSA_ERR_NO_DEVICE, "cache has no device storage");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ErrorWord host{};
  cudaError_t e = cudaMemcpyAsync(&host, c->err(), sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->err(), 0, sizeof host, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *dev_status = host.status;
  if (detail) *detail = host.detail;
  return ok();
}

qsa_status_t qsa_index_score(qsa_cache* c, const qsa_batch* batch, const float* q_idx,
                             const float* w, float* blk_scores, int64_t blk_stride, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  BatchDesc d;
  if (qsa_status_t st = c->build_batch(batch, &d)) return st;
  if (!q_idx || !w || !blk_scores) return fail(QSA_ERR_INVALID_ARG, "null q_idx, w or blk_scores");
  for (int u = 0; u < d.n_units; ++u)
    if (blk_stride < (d.u[u].n + 3) / 4)
      return fail(QSA_ERR_INVALID_ARG, "blk_stride %lld < %lld blocks of unit %d",
                  (long long)blk_stride, (long long)((d.u[u].n + 3) / 4), u);
  cudaError_t e = launch_index_score(d, &c->keys_map, &c->scales_map, q_idx, w, blk_scores, blk_stride,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "index-score launch");
  return ok();
}

qsa_status_t qsa_select_c4_topk(qsa_cache* c, const qsa_batch* batch, const float* blk_scores,
                                int64_t blk_stride, int32_t budget_tokens, int32_t* sel_blocks,
                                int32_t* n_sel, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  BatchDesc d;
  if (qsa_status_t st = c->build_batch(batch, &d)) return st;
  if (!blk_scores || !sel_blocks || !n_sel) return fail(QSA_ERR_INVALID_ARG, "null array");
  if (budget_tokens < 4 || budget_tokens % 4 || budget_tokens > c->cfg.budget_tokens)
    return fail(QSA_ERR_INVALID_ARG, "budget_tokens %d must be a multiple of 4 in [4, %d]",
                budget_tokens, c->cfg.budget_tokens);
  for (int u = 0; u < d.n_units; ++u)
    if (blk_stride < (d.u[u].n + 3) / 4)
      return fail(QSA_ERR_INVALID_ARG, "blk_stride too small for unit %d", u);
  cudaError_t e = launch_select_topk(d, blk_scores, blk_stride, budget_tokens / 4, sel_blocks,
                                     n_sel, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return ok();
}

qsa_status_t qsa_gather_rows(qsa_cache* c, const qsa_batch* batch, const int32_t* sel_blocks,
                             const int32_t* n_sel, int32_t budget_tokens, void* rows_out,
                             int32_t* n_rows, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  BatchDesc d;
  if (qsa_status_t st = c->build_batch(batch, &d)) return st;
  if (!sel_blocks || !n_sel || !rows_out) return fail(QSA_ERR_INVALID_ARG, "null array");
  if (budget_tokens < 4 || budget_tokens % 4 || budget_tokens > c->cfg.budget_tokens)
    return fail(QSA_ERR_INVALID_ARG, "bad budget_tokens %d", budget_tokens);
  if (reinterpret_cast<uintptr_t>(rows_out) % 16)
    return fail(QSA_ERR_INVALID_ARG, "rows_out must be 16-byte aligned");
  cudaError_t e = launch_gather_rows(d, sel_blocks, n_sel, budget_tokens,
                                     static_cast<uint8_t*>(rows_out), n_rows,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  return ok();
}

qsa_status_t qsa_append_token(qsa_cache* c, const qsa_batch* batch, const float* k_new,
                              const void* kv_new, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  BatchDesc d;
  if (qsa_status_t st = c->build_batch(batch, &d)) return st;
  if (!k_new || !kv_new) return fail(QSA_ERR_INVALID_ARG, "null k_new or kv_new");
  if (reinterpret_cast<uintptr_t>(k_new) % 16 || reinterpret_cast<uintptr_t>(kv_new) % 16)
    return fail(QSA_ERR_INVALID_ARG, "k_new and kv_new must be 16-byte aligned");
  AppendTargets tg;
  for (int u = 0; u < d.n_units; ++u) {
    const Lease& l = c->leases[d.u[u].req];
    const int64_t t = l.ctx_len - 1;
    const int64_t layer = d.u[u].layer;
    tg.pool_row[u] = -1;
    tg.evict[u] = -1;
    if (l.placement == QSA_KV_HBM) {
      tg.pool_row[u] = l.row_base + layer * l.layer_rows + t;
    } else if (l.placement == QSA_KV_HOST_RING) {
      tg.pool_row[u] = l.row_base + layer * l.layer_rows + t % l.layer_rows;
      if (t >= l.layer_rows) tg.evict[u] = t - l.layer_rows;
    }
  }
  cudaError_t e = launch_append_token(d, tg, k_new, static_cast<const uint8_t*>(kv_new),
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return ok();
}

qsa_status_t qsa_hot_cache_fetch(qsa_cache* c, const qsa_batch* batch, const int32_t* sel_blocks,
                                 const int32_t* n_sel, int32_t budget_tokens, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  BatchDesc d;
  if (qsa_status_t st = c->build_batch(batch, &d)) return st;
  if (!sel_blocks || !n_sel) return fail(QSA_ERR_INVALID_ARG, "null array");
  if (budget_tokens < 4 || budget_tokens % 4 || budget_tokens > c->cfg.budget_tokens)
    return fail(QSA_ERR_INVALID_ARG, "bad budget_tokens %d", budget_tokens);
  if (c->cfg.hot_rows == 0) return ok();
  cudaError_t e = launch_hot_fetch(d, sel_blocks, n_sel, budget_tokens, true,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "hot-cache launch");
  return ok();
}

qsa_status_t qsa_hot_cache_plan(qsa_cache* c, const qsa_batch* batch, const int32_t* sel_blocks,
                                const int32_t* n_sel, int32_t budget_tokens, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  BatchDesc d;
  if (qsa_status_t st = c->build_batch(batch, &d)) return st;
  if (!sel_blocks || !n_sel) return fail(QSA_ERR_INVALID_ARG, "null array");
  if (budget_tokens < 4 || budget_tokens % 4 || budget_tokens > c->cfg.budget_tokens)
    return fail(QSA_ERR_INVALID_ARG, "bad budget_tokens %d", budget_tokens);
  if (c->cfg.hot_rows == 0) return ok();
  cudaError_t e = launch_hot_fetch(d, sel_blocks, n_sel, budget_tokens, false,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "hot-cache plan launch");
  return ok();
}

qsa_status_t qsa_sparse_decode_attn(qsa_cache* c, const qsa_batch* batch, const uint16_t* q,
                                    const int32_t* sel_blocks, const int32_t* n_sel,
                                    int32_t budget_tokens, const void* gathered,
                                    float softmax_scale, float* out, float* lse, void* stream) {
  if (!c) return fail(QSA_ERR_INVALID_ARG, "null cache");
  DeviceGuard guard(c->device);
  if (qsa_status_t st = c->check_stream(stream, guard)) return st;
  BatchDesc d;
  if (qsa_status_t st = c->build_batch(batch, &d)) return st;
  if (!q || !sel_blocks || !n_sel || !out) return fail(QSA_ERR_INVALID_ARG, "null array");
  if (budget_tokens < 4 || budget_tokens % 4 || budget_tokens > c->cfg.budget_tokens)
    return fail(QSA_ERR_INVALID_ARG, "bad budget_tokens %d", budget_tokens);
  if (reinterpret_cast<uintptr_t>(gathered) % 16 || reinterpret_cast<uintptr_t>(q) % 16)
    return fail(QSA_ERR_INVALID_ARG, "q and gathered must be 16-byte aligned");
  if (!(softmax_scale == softmax_scale)) return fail(QSA_ERR_INVALID_ARG, "softmax_scale is NaN");
  cudaError_t e = launch_sparse_attn(d, q, sel_blocks, n_sel, budget_tokens,
                                     static_cast<const uint8_t*>(gathered), softmax_scale, out,
                                     lse, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return ok();
}

}  // extern "C"
