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
// The scan does 512 multiply-adds per 66 bytes, more than the CUDA cores
// deliver at HBM speed, and it is a genuine dense contraction
// (keys[tokens][64] x q^T[64][8 heads]), so it runs on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM), in tiles of M = 128 tokens.
// The grid is persistent (up to two CTAs per SM) and the work is handed out
// dynamically: CTAs take chunks of the flat tile list of all units of the
// call from an atomic counter, large chunks first and single tiles at the
// end.  A CTA that starts late (its SM busy with another kernel, e.g. the
// attention of other requests on another stream) then simply takes less work
// instead of holding up the whole call with a fixed share.  The last CTA to
// finish re-arms the counter.  Its warps have fixed roles and hand tiles to
// each other through mbarrier rings, so no role waits for another's latency:
//  * TMA warp (lane 0): takes the chunks, streams each tile's 8 KiB of codes
//    into a ring of shared-memory stages with bulk copies (cp.async.bulk;
//    completion counted in bytes on the stage's mbarrier) and publishes the
//    tile's id in a ring read by the MMA warp and the epilogue.
//  * 4 converter warps: turn the codes into the f16 A operand (exact: every
//    e4m3 value is an f16 value); consecutive 16-byte reads, conflict-free
//    stores thanks to the swizzle below.
//  * MMA warp: builds the B operand when the stream enters a new unit - the
//    index query split as q = hi + lo with hi = f16(q), lo = f16(q - hi), rows
//    0-7 and 8-15 of an N = 16 operand, which keeps the dot products at fp32
//    accuracy - and its lane 0 issues four tcgen05.mma per tile (K = 16 each)
//    into one of four 16-column TMEM accumulators, committing to mbarriers
//    that release the A buffer and publish the accumulator.
//  * 2 x 4 epilogue warps (alternate tiles): tcgen05.ld of the tile's 16
//    columns (thread t = token t = TMEM lane t), hi + lo, scale, relu, head
//    weights, C4 max through shuffles, one fp32 per block to global memory.
//
// Operand layout: K-major with the 128-byte swizzle.  A row (one token of A,
// one head of B) is 64 f16 = 128 bytes; its 16-byte chunk c is stored at chunk
// position c ^ (row % 8), so the tensor core reads whole 128-byte lines and
// the converters' stores hit distinct banks.  The descriptor's stride byte
// offset is 1024 (8 rows); K-step k starts 32*k bytes into the row.
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
  int32_t tile_start[kMaxUnits + 1];  // prefix sums of tiles (or CTAs) per unit
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

constexpr int kTcTile = 128;                           // tokens per MMA tile (M)
#ifndef QSA_K1_STAGES
#define QSA_K1_STAGES 4
#endif
#ifndef QSA_K1_CTAS_PER_SM
#define QSA_K1_CTAS_PER_SM 2
#endif
// Register budget per thread: two CTAs at 48 (43 K registers) leave room on
// the SM for one attention CTA.
#ifndef QSA_K1_MAXREG
#define QSA_K1_MAXREG 48
#endif
// Warp roles of the persistent CTA.
constexpr int kWarpTma = 0;                            // lane 0 streams codes with TMA
constexpr int kWarpConv0 = 1;                          // warps 1..4 convert codes to f16
constexpr int kWarpMma = 5;                            // builds B, lane 0 issues the MMAs
constexpr int kWarpEpi0 = 6;                           // warps 6.. read TMEM, score, store
constexpr int kEpiGroups = 2;                          // epilogue groups take alternate tiles
constexpr int kTcThreads = 32 * (kWarpEpi0 + 4 * kEpiGroups);
constexpr int kStages = QSA_K1_STAGES;                 // code ring depth
#ifndef QSA_K1_ABUFS
#define QSA_K1_ABUFS 2
#endif
constexpr int kABufs = QSA_K1_ABUFS;                   // A operand ring
constexpr int kDBufs = 4;                              // TMEM accumulator ring (16 columns each)
constexpr int kIdRing = 16;                            // tile-id ring (producer -> epilogue)
constexpr int kIdReaders = 4;                          // the owning group's 4 warps
constexpr int kRawBytes = kTcTile * kIndexDim;         // 8 KiB of codes per tile
constexpr int kRowBytes128 = kIndexDim * 2;            // one f16 row of A or B: 128 B
constexpr int kABufBytes = kTcTile * kRowBytes128;     // 16 KiB, 1024-aligned
constexpr int kBBytes = 16 * kRowBytes128;             // 2 KiB: rows 0-7 q_hi, rows 8-15 q_lo
constexpr int kBSlotBytes = kBBytes;                   // one unit's B
constexpr uint32_t kTmemCols = 16 * kDBufs;            // 64
constexpr int kCtasPerSm = QSA_K1_CTAS_PER_SM;
constexpr int kOffRaw = 0;
constexpr int kOffA = kOffRaw + kStages * kRawBytes;   // multiple of 1024
constexpr int kOffB = kOffA + kABufs * kABufBytes;
constexpr int kOffBar = kOffB + 2 * kBSlotBytes;
// barriers: raw_full[S], raw_empty[S], a_full[A], a_empty[A], d_full[D],
// d_empty[D], id_full[R], id_empty[R], b_full[2], b_empty[2]
constexpr int kNumBars = 2 * kStages + 2 * kABufs + 2 * kDBufs + 2 * kIdRing + 4;
constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr int kOffStageMeta = kOffTmemSlot + 16;       // int32 [kStages]: run of each stage
constexpr int kOffAMeta = kOffStageMeta + 4 * kStages; // int32 [kABufs]: run of each A buffer
constexpr int kOffIdRing = kOffAMeta + 4 * kABufs;     // int32 [kIdRing]
// + 1 KiB so the operand region can be aligned to 1024 bytes (128-byte swizzle)
constexpr int kTcSmemBytes = kOffIdRing + 4 * kIdRing + 1024;
// kind::f16 instruction descriptor: D f32 (bit 4), A = B = f16, both K-major,
// N/8 at bits 17-22, M/16 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kWaitPolls = 1u << 20;              // bounded mbarrier waits
// Guided chunks: a grab takes 1/kChunkDiv of the unit's remaining tiles per
// CTA sharing it, at most kChunkMax.
#ifndef QSA_K1_CHUNK_DIV
#define QSA_K1_CHUNK_DIV 4
#endif
#ifndef QSA_K1_CHUNK_MAX
#define QSA_K1_CHUNK_MAX 16
#endif
constexpr int kChunkDiv = QSA_K1_CHUNK_DIV;
constexpr int kChunkMax = QSA_K1_CHUNK_MAX;
constexpr int kEndOfWork = -1;                         // tile id that ends a role's loop
constexpr int kWaitFailed = -2;

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return (uint32_t)__cvta_generic_to_shared(ptr);
}

// Byte offset of element (row, k) of a K-major operand with rows of 64 f16
// (128 bytes) under the 128-byte swizzle: 16-byte chunk c of row r is stored
// at chunk position c ^ (r % 8).
__device__ __forceinline__ uint32_t sw128_off(int row, int k) {
  return row * kRowBytes128 + ((((k >> 3) ^ row) & 7) << 4) + (k & 7) * 2;
}

// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: start
// address >> 4, leading byte offset 16 (unused by this layout), stride byte
// offset 1024 (next group of 8 rows), version 1 at bit 46, layout type 2
// (SWIZZLE_128B) at bits 61-63.  K-step k of 16 f16 starts 32*k bytes in.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; false (and an error record) if the phase never completes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, ErrorWord* err,
                                          int64_t detail) {
  for (uint32_t polls = 0; !mbar_try_wait(bar, parity);) {
    if (++polls > kWaitPolls) {
      report_error(err, QSA_ERR_TIMEOUT, kKernIndexScore, detail);
      return false;
    }
  }
  return true;
}

// TMA bulk copy of `bytes` (multiple of 16) from global to shared memory,
// completing `bytes` transactions on mbarrier `bar`.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                            uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
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

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

// Four e4m3 codes (bytes of w, low first) -> two f16x2 words (exact).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ int unit_of_tile(const IndexScoreParams& p, int t) {
  int lo = 0, hi = p.b.n_units - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Work counter of unit u for the current call (the workspace keeps two
// int32 per request x layer; the first counts the unit's tiles handed out).
__device__ __forceinline__ int32_t* unit_counter(const BatchDesc& b, int u) {
  return b.tickets + 2 * ((int64_t)b.u[u].req * b.n_layers + b.u[u].layer);
}

__device__ __forceinline__ int ld_relaxed_gpu(const int32_t* ptr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// Tile range [ts, te) of the unit that holds tile t, cached between calls.
struct UnitCursor {
  int u = -1, ts = 0, te = 0;
  __device__ __forceinline__ bool move_to(const IndexScoreParams& p, int t) {
    if (t >= ts && t < te) return false;
    u = unit_of_tile(p, t);
    ts = p.tile_start[u];
    te = p.tile_start[u + 1];
    return true;
  }
};

__global__ void __maxnreg__(QSA_K1_MAXREG)
index_score_tc_kernel(const IndexScoreParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled operands need 1024-byte alignment
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + kOffBar;
  constexpr int kBarA = 2 * kStages, kBarD = kBarA + 2 * kABufs, kBarId = kBarD + 2 * kDBufs;
  constexpr int kBarB = kBarId + 2 * kIdRing;
  auto raw_full = [&](int i) { return bars + 8u * (uint32_t)i; };
  auto raw_empty = [&](int i) { return bars + 8u * (uint32_t)(kStages + i); };
  auto a_full = [&](int i) { return bars + 8u * (uint32_t)(kBarA + i); };
  auto a_empty = [&](int i) { return bars + 8u * (uint32_t)(kBarA + kABufs + i); };
  auto d_full = [&](int i) { return bars + 8u * (uint32_t)(kBarD + i); };
  auto d_empty = [&](int i) { return bars + 8u * (uint32_t)(kBarD + kDBufs + i); };
  auto id_full = [&](int i) { return bars + 8u * (uint32_t)(kBarId + i); };
  auto id_empty = [&](int i) { return bars + 8u * (uint32_t)(kBarId + kIdRing + i); };
  auto b_full = [&](int i) { return bars + 8u * (uint32_t)(kBarB + i); };
  auto b_empty = [&](int i) { return bars + 8u * (uint32_t)(kBarB + 2 + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  volatile int32_t* stage_meta = reinterpret_cast<volatile int32_t*>(smem + kOffStageMeta);
  volatile int32_t* a_meta = reinterpret_cast<volatile int32_t*>(smem + kOffAMeta);
  volatile int32_t* id_ring = reinterpret_cast<volatile int32_t*>(smem + kOffIdRing);
  const int total = p.tile_start[p.b.n_units];

  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)), "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(raw_full(i), 1); mbar_init(raw_empty(i), 128); }
    for (int i = 0; i < kABufs; ++i) { mbar_init(a_full(i), 128); mbar_init(a_empty(i), 1); }
    for (int i = 0; i < kDBufs; ++i) { mbar_init(d_full(i), 1); mbar_init(d_empty(i), 128); }
    for (int i = 0; i < kIdRing; ++i) { mbar_init(id_full(i), 1); mbar_init(id_empty(i), kIdReaders); }
    for (int i = 0; i < 2; ++i) { mbar_init(b_full(i), 1); mbar_init(b_empty(i), 1); }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ---- producer (whole warp; lane 0 does the atomics, waits and copies).
    // Work comes in chunks of one unit's tiles from that unit's counter; a
    // CTA starts on its home unit (CTAs spread over the units in proportion
    // to their tiles) and stays on a unit until it runs dry, then moves to
    // the unit with the most tiles left.  Chunks shrink as a unit's work runs
    // out, and the next chunk is taken one chunk early.  Consecutive tiles of
    // one unit form a run; for each run the warp writes the unit's B operand
    // into one of two slots.  Each tile's codes go into the ring (with the
    // run number for the converters and the MMA lane) and its flat id into
    // the id ring (for the epilogue).  After the last tile the producer marks
    // the end: one stage for the converters (which pass it on to the MMA
    // lane) and kEpiGroups id slots for the epilogue groups (each group reads
    // ahead to its next own tile).
    const int grid = (int)gridDim.x, n_units = p.b.n_units;
    auto tiles_of = [&](int uu) { return p.tile_start[uu + 1] - p.tile_start[uu]; };
    auto chunk = [&](int uu, int seen) {
      const int64_t share = (int64_t)grid * tiles_of(uu) / total;
      const int c = (int)((tiles_of(uu) - seen) / (kChunkDiv * (share < 1 ? 1 : share)));
      return c < 1 ? 1 : (c > kChunkMax ? kChunkMax : c);
    };
    int u = unit_of_tile(p, (int)((int64_t)blockIdx.x * total / grid));
    int t = 0, t_end = 0;            // current chunk: local tiles [t, t_end) of unit u
    int pref = 0, pref_sz = 0;       // next chunk of unit u (value valid in lane 0)
    bool have_pref = false, first = true, done = false, ok = true;
    int run = -1, run_u = -1;        // current run and its unit
    int64_t n = 0;
    const uint8_t* keys = nullptr;
    int i = 0;
    for (;; ++i) {
      while (t >= t_end) {
        if (have_pref) {
          have_pref = false;
          const int s0 = __shfl_sync(0xFFFFFFFFu, pref, 0);
          if (s0 < tiles_of(u)) {
            t = s0;
            t_end = s0 + pref_sz < tiles_of(u) ? s0 + pref_sz : tiles_of(u);
          }
        } else {
          int uu = u, rem = tiles_of(u);
          if (!first) {
            // the unit with the most tiles left (lowest index on ties)
            uu = -1;
            rem = 0;
            for (int v = lane; v < n_units; v += 32) {
              const int r = tiles_of(v) - ld_relaxed_gpu(unit_counter(p.b, v));
              if (r > rem) { rem = r; uu = v; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const int r2 = __shfl_xor_sync(0xFFFFFFFFu, rem, o);
              const int u2 = __shfl_xor_sync(0xFFFFFFFFu, uu, o);
              if (r2 > rem || (r2 == rem && (unsigned)u2 < (unsigned)uu)) { rem = r2; uu = u2; }
            }
            if (uu < 0) { done = true; break; }
          }
          first = false;
          const int sz = chunk(uu, tiles_of(uu) - rem);
          int s0 = 0;
          if (lane == 0) s0 = atomicAdd(unit_counter(p.b, uu), sz);
          s0 = __shfl_sync(0xFFFFFFFFu, s0, 0);
          if (s0 >= tiles_of(uu)) continue;   // ran dry meanwhile: look again
          u = uu;
          t = s0;
          t_end = s0 + sz < tiles_of(u) ? s0 + sz : tiles_of(u);
        }
        if (t < t_end && t_end < tiles_of(u)) {   // take the next chunk early
          pref_sz = chunk(u, t_end);
          if (lane == 0) pref = atomicAdd(unit_counter(p.b, u), pref_sz);
          have_pref = true;
        }
      }
      if (done) break;
      if (u != run_u) {
        // new run: B operand of unit u into slot run & 1, once the MMAs of
        // run - 2 (the slot's last user) have completed
        ++run;
        run_u = u;
        const int slot = run & 1;
        if (run >= 2) {
          if (lane == 0)
            ok = mbar_wait(b_empty(slot), (uint32_t)((run >> 1) - 1) & 1u, p.b.err, run);
          if (!__shfl_sync(0xFFFFFFFFu, (int)ok, 0)) break;
        }
        uint8_t* B = smem + kOffB + slot * kBSlotBytes;
        const float* qu = p.q_idx + (int64_t)u * kIndexHeads * kIndexDim;
        constexpr int kPerLane = kIndexHeads * kIndexDim / 32;
        float qv[kPerLane];            // all loads in flight before the first store
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) qv[k] = qu[lane + 32 * k];
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int e = lane + 32 * k, h = e >> 6, d = e & 63;
          const __half qh = __float2half_rn(qv[k]);
          const __half ql = __float2half_rn(qv[k] - __half2float(qh));
          *reinterpret_cast<__half*>(B + sw128_off(h, d)) = qh;
          *reinterpret_cast<__half*>(B + sw128_off(h + 8, d)) = ql;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(b_full(slot));
          n = p.b.u[u].n;
          keys = p.b.index_keys + p.b.unit_row(u) * kIndexDim;
        }
      }
      const int tg = p.tile_start[u] + t;      // flat tile id
      if (lane == 0) {
        const int st = i % kStages, rs = i % kIdRing;
        if (i >= kStages) ok = mbar_wait(raw_empty(st), (uint32_t)(i / kStages - 1) & 1u, p.b.err, tg);
        if (ok && i >= kIdRing)
          ok = mbar_wait(id_empty(rs), (uint32_t)(i / kIdRing - 1) & 1u, p.b.err, tg);
        if (ok) {
          id_ring[rs] = tg;
          mbar_arrive(id_full(rs));
          stage_meta[st] = run;
          const int64_t tok0 = (int64_t)t * kTcTile;
          const int64_t left = n - tok0;
          const uint32_t bytes = (uint32_t)((left < kTcTile ? left : kTcTile) * kIndexDim);
          tma_load_1d(sb + kOffRaw + st * kRawBytes, keys + tok0 * kIndexDim, bytes, raw_full(st));
        }
      }
      if (!__shfl_sync(0xFFFFFFFFu, (int)ok, 0)) break;
      ++t;
    }
    if (ok && lane == 0) {
      const int st = i % kStages;
      if (i < kStages || mbar_wait(raw_empty(st), (uint32_t)(i / kStages - 1) & 1u, p.b.err, -1)) {
        stage_meta[st] = kEndOfWork;
        mbar_arrive(raw_full(st));
      }
      for (int j = i; j < i + kEpiGroups; ++j) {
        const int rs = j % kIdRing;
        if (j >= kIdRing && !mbar_wait(id_empty(rs), (uint32_t)(j / kIdRing - 1) & 1u, p.b.err, -1))
          break;
        id_ring[rs] = kEndOfWork;
        mbar_arrive(id_full(rs));
      }
    }
  } else if (warp < kWarpMma) {
    // ---- converters: e4m3 codes -> f16 A operand (exact); the stage's run
    // number travels on with the A buffer
    const int c = tid - 32 * kWarpConv0;  // 0..127
    for (int i = 0;; ++i) {
      const int st = i % kStages, ab = i % kABufs;
      if (!mbar_wait(raw_full(st), (uint32_t)(i / kStages) & 1u, p.b.err, i)) break;
      const int run = stage_meta[st];
      uint4 q[4];
      if (run >= 0) {
        const uint8_t* raw = smem + kOffRaw + st * kRawBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = *reinterpret_cast<const uint4*>(raw + (k * 128 + c) * 16);
        mbar_arrive(raw_empty(st));
      }
      if (i >= kABufs && !mbar_wait(a_empty(ab), (uint32_t)(i / kABufs - 1) & 1u, p.b.err, i))
        break;
      if (c == 0) a_meta[ab] = run;
      if (run < 0) {                  // end of the stream: hand it to the MMA lane
        mbar_arrive(a_full(ab));
        break;
      }
      uint8_t* A = smem + kOffA + ab * kABufBytes;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int lc = k * 128 + c;           // 16-byte chunk of codes in the tile
        const int row = lc >> 2, q16 = lc & 3; // token row, which 16 of its 64 codes
        uint32_t h[8];
        e4m3x4_to_f16x4(q[k].x, h[0], h[1]);
        e4m3x4_to_f16x4(q[k].y, h[2], h[3]);
        e4m3x4_to_f16x4(q[k].z, h[4], h[5]);
        e4m3x4_to_f16x4(q[k].w, h[6], h[7]);
        uint8_t* dst = A + row * kRowBytes128;   // f16 chunks 2*q16 and 2*q16+1, swizzled
        *reinterpret_cast<uint4*>(dst + ((((2 * q16) ^ row) & 7) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + ((((2 * q16 + 1) ^ row) & 7) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(a_full(ab));
    }
  } else if (warp == kWarpMma) {
    // ---- MMA issue, lane 0 alone: per tile four tcgen05.mma (K = 16 each)
    // into a 16-column accumulator; at a new run it releases the previous
    // run's B slot (commit: arrives once those MMAs are done) and waits for
    // the new slot to be written.
    if (lane == 0) {
      int cur_run = -1;
      for (int i = 0;; ++i) {
        const int ab = i % kABufs, db = i % kDBufs;
        if (!mbar_wait(a_full(ab), (uint32_t)(i / kABufs) & 1u, p.b.err, i)) break;
        const int run = a_meta[ab];
        if (run < 0) break;
        if (run != cur_run) {
          if (cur_run >= 0) tc_commit(b_empty(cur_run & 1));
          cur_run = run;
          if (!mbar_wait(b_full(run & 1), (uint32_t)(run >> 1) & 1u, p.b.err, run)) break;
        }
        if (i >= kDBufs && !mbar_wait(d_empty(db), (uint32_t)(i / kDBufs - 1) & 1u, p.b.err, i)) break;
        tc_fence_after();
        const uint32_t a0 = sb + kOffA + ab * kABufBytes;
        const uint32_t b0 = sb + kOffB + (run & 1) * kBSlotBytes;
        const uint32_t d = tmem + (uint32_t)(db * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k)   // columns 0-7: A . q_hi, columns 8-15: A . q_lo
          tc_mma_f16(d, smem_desc_sw128(a0 + 32 * k), smem_desc_sw128(b0 + 32 * k), k > 0 ? 1u : 0u);
        tc_commit(a_empty(ab));
        tc_commit(d_full(db));
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: kEpiGroups groups of 4 warps; group g scores the tiles
    // at stream positions g, g + kEpiGroups, ...  TMEM lane quarter =
    // warp % 4, and the token of the tile = TMEM lane.  Each warp reads the
    // tile ids two own tiles ahead and fetches those tiles' scales early.
    static_assert(kWarpEpi0 == kWarpMma + 1, "warp roles");
    constexpr int G = kEpiGroups;
    const int grp = (warp - kWarpEpi0) >> 2;
    const int qtr = warp & 3;
    const int e = qtr * 32 + lane;
    auto peek = [&](int pos) -> int {
      const int rs = pos % kIdRing;
      int t = kWaitFailed;
      if (lane == 0) {
        if (mbar_wait(id_full(rs), (uint32_t)(pos / kIdRing) & 1u, p.b.err, pos)) t = id_ring[rs];
        if (t >= 0) mbar_arrive(id_empty(rs));
      }
      return __shfl_sync(0xFFFFFFFFu, t, 0);
    };
    UnitCursor sc_cur;                 // unit of the scale cursor
    int64_t sn = 0;
    const uint16_t* sp = nullptr;
    auto scale_of = [&](int t) -> uint16_t {
      if (t < 0) return (uint16_t)0;
      if (sc_cur.move_to(p, t)) {
        sn = p.b.u[sc_cur.u].n;
        sp = p.b.index_scales + p.b.unit_row(sc_cur.u);
      }
      const int64_t tk = (int64_t)(t - sc_cur.ts) * kTcTile + e;
      return tk < sn ? sp[tk] : (uint16_t)0;
    };
    UnitCursor cur;
    int64_t n = 0;
    float* out = nullptr;
    float w[kIndexHeads];
    int idA = peek(grp);
    int idB = idA >= 0 ? peek(grp + G) : kEndOfWork;
    uint16_t scA = scale_of(idA), scB = scale_of(idB);
    for (int i = grp; idA >= 0; i += G) {
      const int t = idA, db = i % kDBufs;
      const int idC = idB >= 0 ? peek(i + 2 * G) : kEndOfWork;
      const uint16_t scC = scale_of(idC);
      if (cur.move_to(p, t)) {
        n = p.b.u[cur.u].n;
        out = p.blk + (int64_t)cur.u * p.blk_stride;
#pragma unroll
        for (int h = 0; h < kIndexHeads; ++h) w[h] = p.w[(int64_t)cur.u * kIndexHeads + h];
      }
      const float sc = __half2float(__ushort_as_half(scA));
      if (!mbar_wait(d_full(db), (uint32_t)(i / kDBufs) & 1u, p.b.err, t)) break;
      tc_fence_after();
      float v[16];
      tc_ld16(tmem + ((uint32_t)(qtr * 32) << 16) + (uint32_t)(db * 16), v);
      tc_fence_before();
      mbar_arrive(d_empty(db));
      const int64_t tok = (int64_t)(t - cur.ts) * kTcTile + e;
      float s = -INFINITY;
      if (tok < n) {
        s = 0.f;
#pragma unroll
        for (int h = 0; h < kIndexHeads; ++h) s = fmaf(w[h], fmaxf((v[h] + v[h + 8]) * sc, 0.f), s);
      }
      s = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
      s = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
      if ((lane & 3) == 0 && tok < n) out[tok >> 2] = s;
      idA = idB; idB = idC;
      scA = scB; scB = scC;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  // the last CTA to finish re-arms the work counters for the next call
  if (tid == 0) {
    int32_t* finished = unit_counter(p.b, 0) + 1;
    __threadfence();
    if (atomicAdd(finished, 1) == (int)gridDim.x - 1) {
      __threadfence();
      for (int uu = 0; uu < p.b.n_units; ++uu) *reinterpret_cast<volatile int32_t*>(unit_counter(p.b, uu)) = 0;
      *reinterpret_cast<volatile int32_t*>(finished) = 0;
    }
  }
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
#ifdef QSA_INDEX_SCORE_FFMA
  const int unit_tokens = kTileTokens;
#else
  const int unit_tokens = kTcTile;
  static bool attr_set = false;
  static int sm_count = 0;
  if (!attr_set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = prefer_max_shared(index_score_tc_kernel, kTcSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
#endif
  int64_t tiles = 0;
  for (int u = 0; u < b.n_units; ++u) {
    p.tile_start[u] = (int32_t)tiles;
    tiles += (b.u[u].n + unit_tokens - 1) / unit_tokens;
  }
  p.tile_start[b.n_units] = (int32_t)tiles;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
#ifdef QSA_INDEX_SCORE_FFMA
  index_score_kernel<<<(unsigned)tiles, kThreads, 0, s>>>(p);
#else
  const int64_t cap = (int64_t)kCtasPerSm * sm_count;
  const unsigned grid = (unsigned)(tiles < cap ? tiles : cap);
  index_score_tc_kernel<<<grid, kTcThreads, kTcSmemBytes, s>>>(p);
#endif
  return cudaGetLastError();
}

}  // namespace qsa
