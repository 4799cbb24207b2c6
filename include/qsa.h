/*
 * qsa.h - C ABI of the QSA sparse-attention decode-step library (one NVIDIA
 * GB300, sm_103a).
 *
 * One decode unit is one request at one QSA layer.  A decode step of a unit:
 *   1. qsa_index_score      score every cached token with the resident
 *                           compact index keys and reduce to C4 block maxima;
 *   2. qsa_select_c4_topk   keep the indexer_budget best tokens, as C4 blocks;
 *   3. qsa_gather_rows      (optional) copy the selected KV rows, found through
 *                           the logical-token -> physical-slot table, into a
 *                           dense buffer;
 *   3a. qsa_hot_cache_fetch (caches with hot rows) copy the selected cold rows
 *                           into the request's hot HBM rows, which keep them
 *                           for later steps, and point their slots there;
 *   4. qsa_sparse_decode_attn  GQA decode attention over the selected rows,
 *                           read through the slot table (HBM rows from the
 *                           pool, cold rows straight from pinned host memory)
 *                           or from the dense buffer of step 3.
 * Producer side: qsa_request_advance reserves the position of a new token and
 * qsa_append_token stores its quantised index key and KV row (per layer,
 * before that layer's step 1).
 * Request leases with generation tags return a finished request's rows and
 * slot-table region to the cache.
 *
 * Sources.  The method is described on two pages:
 *  [offload digest] "Оффлоадинг KV-кэша Qwen3.8-Flash-Next в RAM через vLLM без
 *      потери скорости декодирования": lead paragraph (12 QSA layers,
 *      indexer_budget=2048, 48 MiB moved per step), section "Механизм
 *      гибридного разреженного оффлоадинга" (resident indexer over compact
 *      66-byte keys, only the selected rows cross the bus) and section
 *      "Эффективность и память" (66 vs 2048 bytes per token per layer).
 *  [RTX4090 port] "双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测": opening
 *      explanation of QSA (C4 blocks of 4 adjacent tokens; the 12 sparse
 *      layers select independently) and section "显存账本：热缓存卸载省下约84%"
 *      (full history in pinned host memory, missing blocks fetched on demand,
 *      logical token addresses kept apart from physical cache slots, leases,
 *      generation tags, tail ring buffer, capacity and slots return to their
 *      initial values after requests end).
 *
 * Fixed geometry (this library's reading of the byte counts on the pages):
 *   index key   = 64 FP8-e4m3 codes + 1 fp16 scale   (66 B / token / layer)
 *   index query = 8 heads x 64 fp32, head weights 8 fp32
 *   token score = sum_h w_h * relu(sum_d q[h][d] * scale * e4m3(code[d]))
 *   KV row      = K[4][128] bf16 then V[4][128] bf16  (2048 B / token / layer),
 *                 or in an FP8 cache (qsa_kv_format) E4M3 codes of K and V plus
 *                 8 fp16 scales (1040 B)
 *   query       = 16 heads x 128 bf16, query head h reads KV head h / 4
 *
 * Conventions for every entry point.
 *  - Return a qsa_status_t; QSA_OK is 0.  Nothing aborts, throws across the
 *    ABI, or traps on the device.  On an error qsa_last_error_string() gives a
 *    message (thread-local, valid until the next call on that thread).
 *  - "device" pointers are CUDA device memory (or, where stated, pinned host
 *    memory mapped into the device address space); "host" pointers are
 *    ordinary CPU memory read before the call returns.
 *  - The caller owns every buffer it passes and keeps it alive until the
 *    work enqueued on `stream` (a cudaStream_t, NULL = legacy default stream)
 *    has finished.  The library owns only the opaque qsa_cache metadata.
 *  - Kernels are enqueued asynchronously.  Faults a kernel detects in its
 *    inputs (a slot id outside the pool, a block id outside the context)
 *    are recorded in a device error word inside the workspace; the offending
 *    item is skipped, never accessed.  qsa_poll_error() reads and clears it.
 *  - All device buffers must be 16-byte aligned.
 *  - A qsa_cache is not thread-safe: one host thread at a time.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_ABI_VERSION 4

#define QSA_INDEX_HEADS 8
#define QSA_INDEX_DIM 64
#define QSA_KV_HEADS 4
#define QSA_HEAD_DIM 128
#define QSA_Q_HEADS 16
#define QSA_ROW_BYTES 2048
/* Row of an FP8 KV cache: K codes [4][128] E4M3, V codes [4][128] E4M3, then
 * fp16 scales K[0..3], V[0..3] (value = scale of its head * e4m3(code)). */
#define QSA_ROW_BYTES_FP8 1040
#define QSA_C4 4
/* Largest number of decode units (request x layer pairs) in one call. */
#define QSA_MAX_UNITS 256
/* Largest indexer budget, in tokens. */
#define QSA_MAX_BUDGET_TOKENS 8192
/* Largest hot_rows of a cache (see qsa_cache_config). */
#define QSA_MAX_HOT_ROWS 65536

typedef enum qsa_status_t {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1,   /* bad pointer, size, layer, budget or stride */
  QSA_ERR_CUDA = 2,          /* a CUDA runtime call failed */
  QSA_ERR_STALE_HANDLE = 3,  /* handle's generation is not the live one */
  QSA_ERR_OUT_OF_SLOTS = 4,  /* no free request slot */
  QSA_ERR_CAPACITY = 5,      /* not enough free HBM pool rows, or ctx > capacity */
  QSA_ERR_BAD_SLOT = 6,      /* device: slot id outside [-1, pool rows) or token outside ctx */
  QSA_ERR_TIMEOUT = 7,       /* device: a bounded wait gave up */
  QSA_ERR_BAD_BLOCK = 8,     /* device: selected block id outside the context */
  QSA_ERR_NO_DEVICE = 9      /* the cache was created without device storage */
} qsa_status_t;

/* Where a request's KV rows live. */
typedef enum qsa_kv_placement {
  /* Every row of every layer in the HBM pool (short requests). */
  QSA_KV_HBM = 0,
  /* Full history in pinned host memory; the newest ring_tokens rows of each
   * layer also in an HBM tail ring (token t in ring row t mod ring_tokens). */
  QSA_KV_HOST_RING = 1,
  /* Full history in pinned host memory only; no HBM rows are leased. */
  QSA_KV_HOST = 2
} qsa_kv_placement;

/* Format of the KV rows of a cache (pool, staging, host histories, gathered
 * rows).  BF16: QSA_ROW_BYTES-byte rows, K[4][128] then V[4][128] bf16.
 * FP8: QSA_ROW_BYTES_FP8-byte rows (layout above), each of the 8 head
 * vectors quantised like an index key: fp16 scale = round-to-nearest-even
 * of absmax/448, codes = E4M3 of clamp(x/scale, +-448) (this library's
 * reading of the FP8 KV cache the RTX 5090 page runs; the RTX4090 port's
 * per-card memory figure fits about 1 KiB per token and layer). */
typedef enum qsa_kv_format {
  QSA_KV_BF16 = 0,
  QSA_KV_FP8 = 1
} qsa_kv_format;

typedef struct qsa_cache_config {
  int32_t n_layers;        /* QSA layers managed per request (e.g. 12) */
  int32_t max_requests;    /* request slots */
  int64_t ctx_capacity;    /* largest context of a request, in tokens */
  int32_t budget_tokens;   /* largest indexer budget; multiple of 4, <= QSA_MAX_BUDGET_TOKENS */
  int32_t ring_tokens;     /* tail ring length per offloaded request and layer (> 0) */
  int32_t staging_rows;    /* shared staging rows per layer, carved from the pool front */
  int32_t kv_format;       /* qsa_kv_format; row bytes R = QSA_ROW_BYTES or QSA_ROW_BYTES_FP8 */
  int64_t hbm_pool_rows;   /* rows of R bytes in hbm_pool */
  /* Device storage (all caller-allocated, 16-byte aligned).  Leave every one
   * NULL for a host-only cache: the bookkeeping entry points then work
   * without a GPU and the compute entry points return QSA_ERR_NO_DEVICE. */
  void* hbm_pool;          /* device [hbm_pool_rows][R]: staging, rings, resident rows */
  uint8_t* index_keys;     /* device [max_requests][n_layers][ctx_capacity][64] e4m3 codes */
  uint16_t* index_scales;  /* device [max_requests][n_layers][ctx_capacity] fp16 bits */
  int32_t* slot_table;     /* device [max_requests][n_layers][ctx_capacity] int32 */
  void* workspace;         /* device, qsa_workspace_bytes(config) bytes */
  int64_t workspace_bytes;
  /* Cross-step hot cache: pool rows per offloaded request and layer that keep
   * cold rows fetched by qsa_hot_cache_fetch for later steps.  0: no hot
   * cache; else budget_tokens <= hot_rows <= QSA_MAX_HOT_ROWS. */
  int32_t hot_rows;
  int32_t reserved1;       /* must be 0 */
} qsa_cache_config;

typedef struct qsa_handle {
  uint32_t index;          /* request slot */
  uint32_t generation;     /* lease generation; stale generations are rejected */
} qsa_handle;

typedef struct qsa_request_desc {
  int64_t ctx_len;         /* cached tokens, 1 <= ctx_len <= ctx_capacity */
  int32_t placement;       /* qsa_kv_placement */
  /* Largest context the request may grow to with qsa_request_advance
   * (ctx_len <= max_ctx <= ctx_capacity); 0 means ctx_len (no growth).  It
   * sets the request's row stride M = max(ctx_len, max_ctx): a QSA_KV_HBM
   * request leases n_layers * M pool rows, and a host history is laid out
   * [n_layers][M][R]. */
  int32_t max_ctx;
  /* QSA_KV_HOST_RING, QSA_KV_HOST: host memory [n_layers][M][R] holding the
   * full history: memory from qsa_host_alloc for this cache's device, or
   * pinned memory registered or allocated with the CUDA runtime's mapped
   * flag (host address; the library finds the device address, and
   * qsa_append_token writes the rows of new tokens into it).
   * QSA_KV_HBM: NULL. */
  const void* host_rows;
} qsa_request_desc;

typedef struct qsa_request_info {
  int64_t ctx_len;
  int32_t placement;
  int32_t layer_rows;      /* pool rows per layer in the request's region */
  int64_t hbm_row_base;    /* first pool row of the region; layer l starts at
                              hbm_row_base + l * layer_rows */
  const void* host_rows;   /* device-usable address of the host history, or NULL */
  int64_t max_ctx;         /* the request's row stride M (see qsa_request_desc) */
  int64_t hot_row_base;    /* first hot row (layer l: hot_row_base + l * hot_rows), or -1
                              when the request has none */
} qsa_request_info;

typedef struct qsa_stats {
  int32_t max_requests;
  int32_t active_requests;
  int32_t free_request_slots;
  int32_t free_ranges;          /* fragments in the pool's free list */
  int64_t hbm_pool_rows;
  int64_t free_hbm_rows;        /* rows not leased to any request (staging excluded) */
  int64_t largest_free_rows;
  int64_t staging_rows_total;   /* n_layers * staging_rows */
  int64_t hbm_kv_bytes_in_use;  /* pool rows leased to requests (ring, resident and hot rows) x R */
} qsa_stats;

/* A batch of decode units: n_req requests at layers layer0 .. layer0+n_layers-1.
 * Unit u = i_layer * n_req + i_req; per-unit arrays are indexed by u. */
typedef struct qsa_batch {
  int32_t n_req;
  int32_t layer0;
  int32_t n_layers;
  int32_t reserved0;
  const qsa_handle* requests;   /* host [n_req] */
} qsa_batch;

typedef struct qsa_cache qsa_cache;

/* ------------------------------------------------------------- lifecycle */

int32_t qsa_abi_version(void);
const char* qsa_last_error_string(void);

/* Bytes of device workspace a cache with this config needs (error word,
 * split-K partials of every request x layer, two int32 work counters per
 * request x layer for qsa_index_score, and with hot_rows > 0 the hot-cache
 * state of every request x layer: a fill list of budget_tokens entries, its
 * length, the cursor, hot_rows owner entries, and the budget_tokens rows and
 * the flag of qsa_hot_cache_plan's pending map).  Returns -1 on a bad
 * config. */
int64_t qsa_workspace_bytes(const qsa_cache_config* config);

/* Create a cache.  Checks the config; with device storage, also zeroes the
 * workspace and marks every slot-table entry cold (synchronously, on the
 * current device).  *out receives the cache; free it with qsa_cache_destroy.
 * Errors: INVALID_ARG (bad sizes, partial device storage, short workspace),
 * CAPACITY (staging does not fit the pool), CUDA. */
qsa_status_t qsa_cache_create(const qsa_cache_config* config, qsa_cache** out);
qsa_status_t qsa_cache_destroy(qsa_cache* cache);

/* ------------------------------------------- leases, slots, bookkeeping */

/* Lease a request slot and an HBM region (M = max(ctx_len, max_ctx) rows
 * per layer for QSA_KV_HBM, ring_tokens rows per layer for
 * QSA_KV_HOST_RING, none for QSA_KV_HOST; with hot_rows > 0 an offloaded
 * request also gets hot_rows rows per layer after its ring rows, all of
 * them free, with the hot-cache cursor at row 0), bump the
 * slot's generation, and enqueue on `stream` the fill of the request's
 * slot-table rows: resident token t of layer l -> region row l*layer_rows + t;
 * offloaded token t -> ring row l*ring_tokens + t mod ring_tokens when t is
 * among the newest ring_tokens tokens, else -1 (cold, read from host_rows);
 * every token of a QSA_KV_HOST request -> -1.
 * [RTX4090 port, memory-ledger section: leases, generation tags, tail ring,
 * logical addresses separate from physical slots.]
 * Errors: INVALID_ARG, CAPACITY (ctx_len or max_ctx > ctx_capacity, or no pool range),
 * OUT_OF_SLOTS, CUDA.  On error nothing is leased. */
qsa_status_t qsa_request_begin(qsa_cache* cache, const qsa_request_desc* desc,
                               void* stream, qsa_handle* out);

/* Return the request's slot and HBM region to the cache.  The handle, and
 * any copy of it, is stale afterwards.  Work already enqueued for it must
 * have finished before its rows are leased again.
 * Errors: STALE_HANDLE (wrong generation, already ended, or index out of
 * range).  [RTX4090 port: finished or cancelled requests give back their KV
 * capacity and cache slots.] */
qsa_status_t qsa_request_end(qsa_cache* cache, qsa_handle handle);

/* The lease of a live request: context length, placement, its pool region
 * (hbm_row_base, layer_rows, hot_row_base), the device-usable address of its
 * host history and its row stride max_ctx.  Errors: INVALID_ARG (null),
 * STALE_HANDLE. */
qsa_status_t qsa_request_info_get(qsa_cache* cache, qsa_handle handle, qsa_request_info* out);

/* Counters of free and leased capacity; equal to their initial values once
 * every request has ended. */
qsa_status_t qsa_cache_stats(const qsa_cache* cache, qsa_stats* out);

/* Device row of the slot table of (request, layer): int32 [ctx_len], valid
 * while the lease lives.  Errors: STALE_HANDLE, INVALID_ARG, NO_DEVICE. */
qsa_status_t qsa_slot_table_ptr(qsa_cache* cache, qsa_handle handle, int32_t layer, int32_t** out);

/* Remap n logical tokens of (request, layer): slot_table[tokens[i]] =
 * slots[i] (device arrays of n int64 / int32), enqueued on stream.  A slot
 * must be -1 (cold: host row) or a pool row; a token must be < ctx_len.
 * Entries that break this are skipped and reported through the device
 * error word (BAD_SLOT).  The caller keeps row contents consistent. */
qsa_status_t qsa_slot_table_set(qsa_cache* cache, qsa_handle handle, int32_t layer,
                                const int64_t* tokens, const int32_t* slots, int32_t n,
                                void* stream);

/* Device pointer to the staging rows of a layer inside the pool
 * ([staging_rows][R]); a landing zone for qsa_gather_rows. */
qsa_status_t qsa_staging_ptr(qsa_cache* cache, int32_t layer, void** out);

/* Read and clear the device error word (synchronises `stream`).
 * *dev_status receives a qsa_status_t recorded by a kernel (QSA_OK if none)
 * and *detail the offending value. */
qsa_status_t qsa_poll_error(qsa_cache* cache, void* stream, int32_t* dev_status, int64_t* detail);

/* ---------------------------------------------------- producer side */

/* Reserve the positions of n_new new tokens of a request: they are
 * ctx_len .. ctx_len + n_new - 1, and ctx_len grows by n_new.  Host
 * bookkeeping only (no device work).  In a decode step call it once, before
 * the step; then store the new token at every layer with qsa_append_token
 * before that layer's qsa_index_score, since until then the new position's
 * key, row and slot are unset.  QSA_ERR_CAPACITY beyond the request's
 * max_ctx, QSA_ERR_INVALID_ARG for n_new < 1, QSA_ERR_STALE_HANDLE for a
 * stale handle; nothing changes on error. */
qsa_status_t qsa_request_advance(qsa_cache* cache, qsa_handle request, int32_t n_new);

/* Store the newest token (position t = ctx_len - 1) of every unit u of the
 * batch (request r, layer l), as the producer side of the decode step
 * ("Оффлоадинг KV-кэша Qwen3.8-Flash-Next в RAM через vLLM без потери
 * скорости декодирования", section "Эффективность и память": 66-byte index
 * key and 2048-byte row per token and layer; "双卡RTX4090跑通Qwen3-Next：
 * 8并发满血长上下文实测", section "显存账本：热缓存卸载省下约84%": full history
 * in pinned host memory, newest tokens in the HBM tail ring, logical tokens
 * kept apart from physical slots).
 *   k_new   device fp32 [units][64]: the token's index key.  Stored as
 *           scale = binary16 round-to-nearest-even of (absmax / 448), the
 *           division in fp32, saturating at 65504; codes = E4M3
 *           round-to-nearest-even of clamp(k / scale, -448, 448), the
 *           division in fp32; a zero scale stores 64 zero codes.
 *   kv_new  device [units][2048]: the token's KV row (K[4][128] then
 *           V[4][128], bf16); stored unchanged in a BF16 cache, quantised
 *           to an FP8 row (QSA_ROW_BYTES_FP8, rule of qsa_kv_format) in an
 *           FP8 cache.
 * Where the row goes, by placement, and the slot-table writes:
 *   QSA_KV_HBM        pool row hbm_row_base + l*M + t; slot[t] = that row.
 *   QSA_KV_HOST       host history row (l, t); slot[t] = -1.
 *   QSA_KV_HOST_RING  host history row (l, t) and ring row
 *                     hbm_row_base + l*ring_tokens + t mod ring_tokens;
 *                     slot[t] = that ring row, and the token that held it,
 *                     t - ring_tokens (if >= 0), becomes cold: slot = -1.
 * Both buffers 16-byte aligned.  Every unit needs ctx_len >= 1. */
qsa_status_t qsa_append_token(qsa_cache* cache, const qsa_batch* batch, const float* k_new,
                              const void* kv_new, void* stream);

/* ------------------------------------------------------------ hot path */

/* Steps 1 and 2a.  For every unit u of the batch (request r, layer l,
 * n = ctx_len tokens): S_t = sum_h w[u][h] * relu(sum_d q_idx[u][h][d] *
 * scale_t * e4m3(code_t[d])) over the resident keys of (r, l), then
 * blk_scores[u * blk_stride + b] = max(S_4b .. S_4b+3) for b < ceil(n/4)
 * (a ragged last block takes the max of the tokens it has).
 * [offload digest, "Механизм гибридного разреженного оффлоадинга": the
 * resident indexer scores every cached token from 66-byte keys; RTX4090 port,
 * opening explanation: C4 blocks of 4 adjacent tokens.]
 * q_idx: device fp32 [units][8][64]; w: device fp32 [units][8];
 * blk_scores: device fp32 [units][blk_stride], blk_stride >= ceil(ctx/4) of
 * every unit.  The CTAs take 128-token tiles from a work counter in the
 * workspace that belongs to the batch's first unit (its request and layer)
 * and reset it when the last CTA ends: two calls that overlap on the GPU and
 * share their first unit race.
 * Errors: INVALID_ARG, STALE_HANDLE, NO_DEVICE, CUDA. */
qsa_status_t qsa_index_score(qsa_cache* cache, const qsa_batch* batch,
                             const float* q_idx, const float* w,
                             float* blk_scores, int64_t blk_stride, void* stream);

/* Step 2b.  Per unit, the K = min(budget_tokens/4, ceil(n/4)) blocks that
 * rank highest under (score descending, block id ascending), written in
 * ascending id order to sel_blocks[u * (budget_tokens/4) + i], with
 * n_sel[u] = K.  -0.0 ranks equal to +0.0.  Scores must not be NaN.
 * [offload digest lead: at most indexer_budget=2048 positions; RTX4090
 * port: selection by C4 block, independently per layer.]
 * blk_scores: device fp32 [units][blk_stride]; sel_blocks: device int32
 * [units][budget_tokens/4]; n_sel: device int32 [units].
 * budget_tokens: multiple of 4, 4 <= budget_tokens <= config budget_tokens. */
qsa_status_t qsa_select_c4_topk(qsa_cache* cache, const qsa_batch* batch,
                                const float* blk_scores, int64_t blk_stride,
                                int32_t budget_tokens, int32_t* sel_blocks, int32_t* n_sel,
                                void* stream);

/* Step 3.  Copy the rows of the selected tokens (tokens 4b..4b+3 of each
 * selected block b, clipped to ctx_len, in that order) into rows_out[u *
 * budget_tokens + i] (2048 B each).  The source of token t of (r, l) is pool
 * row slot_table[t] when that is >= 0, else row t of the request's pinned
 * host history for layer l.  n_rows[u] (device, may be NULL) receives the
 * row count.  [RTX4090 port, memory-ledger section: missing blocks are moved
 * back from pinned host memory on demand; offload digest: only the selected
 * rows cross the bus.]  rows_out: device [units][budget_tokens][R] (R: the
 * cache's row bytes). */
qsa_status_t qsa_gather_rows(qsa_cache* cache, const qsa_batch* batch,
                             const int32_t* sel_blocks, const int32_t* n_sel,
                             int32_t budget_tokens, void* rows_out, int32_t* n_rows,
                             void* stream);

/* Step 3a (caches with hot_rows > 0).  Cross-step hot cache: per unit of
 * an offloaded request, move the rows of the selected tokens that are cold
 * (slot -1) from pinned host memory into the unit's hot rows and point their
 * slots there, so that qsa_gather_rows and qsa_sparse_decode_attn read every
 * selected row from HBM, and rows fetched in one step serve later steps.
 * [RTX4090 port, memory-ledger section: the full history stays in pinned
 * host memory and missing blocks are moved back to the GPU on demand, into a
 * hot cache found through the slot table.]  Replacement (this library's
 * reading; the page names no rule): for the selected tokens (tokens 4b ..
 * 4b+3 of each selected block, clipped to ctx_len), a token whose slot is
 * one of the unit's hot rows is a hit and its row is in use by this step; the
 * cold ones (misses) take rows in ascending token order; the rows handed out
 * are the first rows not in use by this step in circular order from the
 * unit's cursor, which then moves one past the last row handed out; the
 * token a handed-out row held becomes cold (slot -1) if its slot still names
 * that row.  Since hot_rows >= budget_tokens, every miss gets a row.
 * Tokens whose slot is another pool row (tail ring, staging) are untouched.
 * Units of QSA_KV_HBM requests, and every unit of a cache without hot rows,
 * are skipped.  sel_blocks/n_sel: as written by qsa_select_c4_topk (ascending
 * distinct blocks).  Two launches per call (a plan kernel, one CTA per unit,
 * and a copy kernel); nothing else may write the same units' slot tables
 * (qsa_append_token, qsa_slot_table_set) while they run.
 * Errors: INVALID_ARG, STALE_HANDLE, NO_DEVICE, CUDA; bad blocks and slots
 * go to the device error word (BAD_BLOCK, BAD_SLOT). */
qsa_status_t qsa_hot_cache_fetch(qsa_cache* cache, const qsa_batch* batch,
                                 const int32_t* sel_blocks, const int32_t* n_sel,
                                 int32_t budget_tokens, void* stream);

/* The plan of qsa_hot_cache_fetch without its copy: the same slot-table,
 * owner and cursor updates (one launch, one CTA per unit), and a per-unit
 * map from selected position to the hot row its miss was given.  The next
 * qsa_sparse_decode_attn of those units (without `gathered`, and with the
 * same sel_blocks and n_sel) reads the misses' rows from host memory, as a
 * zero-copy read would, and writes them into their hot rows as it goes;
 * afterwards the units are in the state qsa_hot_cache_fetch leaves.  Until that attention has run, the misses'
 * hot rows hold stale bytes: no other call may read those units' rows
 * (qsa_gather_rows, attention with `gathered`), and the pending map is
 * replaced by the next plan or fetch of the unit.
 * [RTX4090 port, memory-ledger section: missing blocks moved back on
 * demand; here the move rides on the attention's own read.]
 * Errors: as qsa_hot_cache_fetch. */
qsa_status_t qsa_hot_cache_plan(qsa_cache* cache, const qsa_batch* batch,
                                const int32_t* sel_blocks, const int32_t* n_sel,
                                int32_t budget_tokens, void* stream);

/* Step 4.  GQA decode attention of each unit over its selected tokens:
 * for query head h (KV head g = h/4), logits_i = softmax_scale * q[u][h] .
 * K_i[g], out[u][h] = sum_i softmax(logits)_i V_i[g], lse[u][h] =
 * log sum_i exp(logits_i) (natural log; -inf and out = 0 with no tokens).
 * Rows come from `gathered` ([units][budget_tokens][R], as written by
 * qsa_gather_rows) when it is not NULL, else through the slot table exactly
 * as qsa_gather_rows reads them (pool rows from HBM, cold rows zero-copy
 * from pinned host memory).  A launch that reads cold rows from host memory
 * is held to a few dozen CTAs, which saturate the host link without slowing
 * HBM-bound work beside it; units with hot rows count as reading only HBM
 * (call qsa_hot_cache_fetch or qsa_hot_cache_plan first; after a plan, this
 * call also copies the planned misses into their hot rows).  Split-K over the tokens with a log-sum-exp merge;
 * partials live in the workspace, per (request, layer): two calls that
 * overlap on the GPU and share a (request, layer) race.
 * [offload digest: attention reads only the <= 2048 selected rows.]
 * q: device bf16 bits [units][16][128]; out: device fp32 [units][16][128];
 * lse: device fp32 [units][16] (may be NULL). */
qsa_status_t qsa_sparse_decode_attn(qsa_cache* cache, const qsa_batch* batch,
                                    const uint16_t* q, const int32_t* sel_blocks,
                                    const int32_t* n_sel, int32_t budget_tokens,
                                    const void* gathered, float softmax_scale,
                                    float* out, float* lse, void* stream);

/* -------------------------------------------------- host history memory */

/* Host memory for the history of offloaded requests, laid out for the device
 * to read selected rows from it: physical pages on host NUMA node numa_node
 * (-1: the node the driver reports as closest to `device`), created and
 * mapped with the driver's virtual-memory API in 2 MiB pieces into one
 * virtual range that the device's own page tables and the host's page
 * tables both hold, at the same address.  Pages that are only registered
 * with cudaHostRegister are reached, on an NVLink-C2C system, through the
 * CPU's page tables one 64 KiB page at a time: read faster while the GPU's
 * cached translations of them are warm, but any munmap in the process (an
 * allocator returning memory) drops those translations, an idle GPU lets
 * them go stale, and a step that touches new pages pays for each; memory
 * from this call reads slower (~70 GB/s of random rows on a GB300 against
 * up to ~186 GB/s) but at the same rate whatever the process does.  bytes
 * is rounded up to 2 MiB.  Pass the address as qsa_request_desc.host_rows of a cache whose
 * storage is on `device`; the host reads and writes the memory like any
 * other.  Free it with qsa_host_free once no request uses it.
 * [RTX4090 port, memory-ledger section: the full history stays in pinned
 * host memory, missing blocks come back to the GPU on demand.]
 * Errors: INVALID_ARG (null out, bytes <= 0, bad device), CAPACITY (no
 * room on the node), CUDA (no virtual-memory API or host NUMA memory). */
qsa_status_t qsa_host_alloc(int32_t device, int32_t numa_node, int64_t bytes, void** out);

/* Unmap and free memory from qsa_host_alloc (NULL: nothing to do).  No
 * request may still use it and no work reading it may be in flight.
 * Errors: INVALID_ARG (not an address qsa_host_alloc returned), CUDA. */
qsa_status_t qsa_host_free(void* ptr);

/* ------------------------------------------- no-allocation variant */

/* Limits of qsa_sparse_decode_attn_noalloc (its scratch is a fixed 8.5 MB
 * device array of this library: 16 units x 64 splits of 32 rows). */
#define QSA_STATIC_MAX_UNITS 16
#define QSA_STATIC_MAX_ROWS 2048

/* Decode attention over dense gathered rows that needs no device memory from
 * the caller beyond its inputs and outputs.  The pages have no counterpart
 * of this entry point; it exists for callers that cannot allocate device
 * memory where they run attention (a serving engine whose device memory is
 * carved from a pre-planned arena it may not grow, a plug-in handed only its
 * input and output buffers, code that must not call cudaMalloc because it
 * would synchronise the device).  It computes what qsa_sparse_decode_attn
 * computes when given gathered rows (equal up to rounding: the splits are
 * merged in another order), without a qsa_cache: the
 * split-K partials live in a static 8.5 MB device array of the library that
 * every GPU which loads the library holds until the process exits.
 *  q:      device bf16 bits [n_units][16][128]
 *  rows:   device [n_units][rows_stride][2048] BF16 rows, as written by qsa_gather_rows
 *          (rows_stride = budget_tokens there); row i of unit u is used when
 *          i < n_rows[u]
 *  n_rows: device int32 [n_units], clamped on the device to [0, rows_stride]
 *  out, lse: as for qsa_sparse_decode_attn (lse may be NULL)
 * Limits: 1 <= n_units <= QSA_STATIC_MAX_UNITS and 1 <= rows_stride <=
 * QSA_STATIC_MAX_ROWS; larger calls return QSA_ERR_INVALID_ARG (split the
 * batch).  No cudaMalloc, cudaFree or allocating library call is made.  The
 * first call on each device looks up the array's device address with
 * cudaGetSymbolAddress (with that device current) and sets the kernel's
 * shared-memory limit; make that first call before any stream capture.
 * Every call shares the one array and leaves its partials there; nothing in
 * it needs to start at zero, because each call writes every partial it reads.
 * Two calls whose work overlaps on the GPU (different streams, or concurrent
 * host threads) race on the array: serialise them. */
qsa_status_t qsa_sparse_decode_attn_noalloc(const uint16_t* q, const void* rows,
                                            const int32_t* n_rows, int32_t n_units,
                                            int32_t rows_stride, float softmax_scale,
                                            float* out, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
