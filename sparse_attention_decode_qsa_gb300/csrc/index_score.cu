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
// tensor cores (tcgen05, kind::f8f6f4): per tile of M = 128 tokens,
// D[128][48] = A . B^T with
//  * A = the tile's e4m3 codes exactly as TMA lands them: 128 rows of 64
//    bytes under the 64-byte swizzle, which is the tensor core's K-major
//    SWIZZLE_64B layout, so the codes are never touched by a thread;
//  * B = the index query as e4m3 "pieces": q * 2^s = sum_p piece_p * 16^-p
//    (p = 0..5; each piece the round-to-nearest e4m3 of the remaining
//    residual times 16), one B row per (piece, head): 6 x 8 = 48 rows, the
//    MMA's N.  An e4m3 rounding leaves a residual of at most 2^-4 of its
//    input, so after six pieces an element's remaining error is at most
//    2^-24 of the element (or, once a residual falls into the e4m3
//    subnormals, at most 2^-37 of the unit's largest element, which the
//    common scale puts in [128, 256)): the pieces carry the fp32 query to
//    fp32's own precision.  Every product of two
//    e4m3 values is exact, and the tensor core accumulates in fp32, so
//    sum_p 16^-p * D[:, 8p + h] / 2^s is the dot product to fp32 rounding.
// Per tile that is two MMAs (K = 32 each); a tensor core spends ~160 cycles
// on an MMA of this size whatever its N, so the instruction count per token
// is what bounds the kernel, and fp8 operands halve it against f16 ones.
//
// The grid is persistent (two CTAs per SM).  Work is handed out in chunks of
// kChunk consecutive tiles of the call's flat tile list from a counter in the
// workspace, so a CTA that starts late (its SM busy with another kernel, e.g.
// the attention of other requests on another stream) takes less work instead
// of holding up the call; the last CTA to finish re-arms the counter.  Warp
// roles, handing tiles over through mbarrier rings (all waits bounded):
//  * producer warp: takes chunks (lane 0, one chunk ahead), builds a group's
//    B operand when the group's stream of tiles enters a new unit (a "run";
//    two B slots per group), issues the TMA loads of each tile (codes, and
//    the tile's fp16 scales) and publishes the tile's (unit, tile, run)
//    in the stage's metadata.
//  * two MMA warps, one per worker group (the first also allocates tensor
//    memory): lane 0 issues the tile's two tcgen05.mma, A and B from shared
//    memory, into one of four accumulators, then releases the stage.
//  * two groups of 4 worker warps, taking alternate tiles: thread = token row
//    = tensor-memory lane.  Each reads its token's scale, then its row of
//    the accumulator, and computes relu, head weights, scale and the C4 max
//    (shuffles); one fp32 per block goes to global memory.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kTile = 128;                      // tokens per tile (MMA M)
#ifndef QSA_K1_PIPES
#define QSA_K1_PIPES 2
#endif
constexpr int kPipes = QSA_K1_PIPES;            // independent pipelines per CTA
#ifndef QSA_K1_STAGES
#define QSA_K1_STAGES 3
#endif
constexpr int kStages = QSA_K1_STAGES;          // code ring depth per pipeline (8 KiB each)
#ifndef QSA_K1_PIECES
#define QSA_K1_PIECES 6
#endif
constexpr int kPieces = QSA_K1_PIECES;          // e4m3 pieces of the query (5 or 6)
constexpr int kN = 48;                          // B rows: 8 heads x 6 pieces (5 pieces: padded)
constexpr int kDBufs = 2;                       // accumulators per pipeline in tensor memory
constexpr int kDStride = 64;                    // tensor-memory columns per accumulator
// Warp roles within a pipeline (6 warps): producer, MMA, 4 workers.
constexpr int kPipeWarps = 6;
constexpr int kRoleProd = 0, kRoleMma = 1, kRoleWork0 = 2;
constexpr int kThreadsTc = 32 * kPipeWarps * kPipes;   // 384
#ifndef QSA_K1_CTAS_PER_SM
#define QSA_K1_CTAS_PER_SM 2
#endif
constexpr int kCtasPerSm = QSA_K1_CTAS_PER_SM;
// Register budget per thread: two CTAs of 12 warps at 56 (43008 registers)
// leave room for one attention CTA (20480) on the SM, and no third CTA of
// this kernel fits (so two always find their tensor memory free).
#ifndef QSA_K1_MAXREG
#define QSA_K1_MAXREG 56
#endif
#ifndef QSA_K1_CHUNK
#define QSA_K1_CHUNK 2   // measured against 1, 4, 8, 16 (8 x 262144 tokens: 30.6 / 26.9 / 27.4 / 28.8 / 29.0 us)
#endif
constexpr int kChunk = QSA_K1_CHUNK;            // tiles per grab from a unit's work counter
constexpr int kRawBytes = kTile * kIndexDim;    // 8 KiB of codes per tile
constexpr int kBBytes = 1024 * ((kN * kIndexDim + 1023) / 1024);   // 3 KiB of pieces
constexpr int kBSlots = 2;                      // per pipeline: current and next run
constexpr uint32_t kPipeCols = kDBufs * kDStride;                  // 128
constexpr uint32_t kTmemCols = kPipeCols * kPipes;                 // 256
// Scales of a tile come with its codes: a 1-D TMA box of kScaleBox fp16
// values starting at the tile's first scale rounded down to a multiple of 8
// (TMA starts on 16-byte boundaries), so the tile's 128 scales sit at an
// offset of 0..7 values into the box.
constexpr int kScaleBox = kTile + 8;            // 136 values = 272 bytes
constexpr int kScaleSlot = 384;                 // bytes per stage, 128-aligned
// Shared memory of one pipeline (1024-aligned stages and B slots first).
constexpr int kOffRaw = 0;
constexpr int kOffB = kOffRaw + kStages * kRawBytes;
constexpr int kOffScale = kOffB + kBSlots * kBBytes;
constexpr int kOffBar = kOffScale + kStages * kScaleSlot;
// barriers: full[S], empty[S], d_full[D], d_empty[D], b_full[B], b_empty[B], mma_done
constexpr int kNumBars = 2 * kStages + 2 * kDBufs + 2 * kBSlots + 1;
constexpr int kOffStageMeta = (kOffBar + 8 * kNumBars + 15) / 16 * 16;   // int4 [kStages]
constexpr int kPipeBytes = (kOffStageMeta + 16 * kStages + 1023) / 1024 * 1024;
constexpr int kOffTmemSlot = kPipes * kPipeBytes;
// + 1 KiB so the pipelines can be aligned to 1024 bytes
constexpr int kSmemBytes = kOffTmemSlot + 16 + 1024;
static_assert(kRawBytes % 1024 == 0 && kOffB % 1024 == 0 && kBBytes % 1024 == 0 &&
                  kPipeBytes % 1024 == 0, "swizzled operands need 1024-byte alignment");
static_assert(kOffScale % 128 == 0 && kScaleSlot % 128 == 0 && kScaleBox * 2 <= kScaleSlot &&
                  (kScaleBox * 2) % 16 == 0, "scale boxes: 16-byte multiples in 128-byte slots");
static_assert(kOffBar % 8 == 0 && kOffStageMeta % 16 == 0,
              "mbarriers need 8-byte, int4 metadata 16-byte alignment");
static_assert((kPieces == 5 || kPieces == 6) && kPieces * kIndexHeads <= kN && kN % 16 == 0 &&
                  kN <= kDStride, "B rows");
static_assert(kPipeWarps - kRoleWork0 == 4, "four worker warps cover the four lane quarters");
// kind::f8f6f4 instruction descriptor: D f32 (bit 4), A = B = e4m3 (type 0 at
// bits 7-9 and 10-12), both K-major, N/8 at bits 17-22, M/16 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kWaitPolls = 1u << 20;       // bounded mbarrier waits
constexpr int kEndOfWork = -1;
constexpr int kRunBits = 20;                    // stage meta .z = run | (s + 1024) << 20

struct IndexScoreParams {
  CUtensorMap keys_map;               // uint8 [rows][64], box 64 x 128, 64-byte swizzle
  CUtensorMap scales_map;             // fp16 [rows], box kScaleBox
  BatchDesc b;
  int32_t tile_start[kMaxUnits + 1];  // prefix sums of tiles per unit
  const float* q_idx;                 // [units][8][64]
  const float* w;                     // [units][8]
  float* blk;                         // [units][blk_stride]
  int64_t blk_stride;
};

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return (uint32_t)__cvta_generic_to_shared(ptr);
}

// Shared-memory matrix descriptor, K-major with the 64-byte swizzle (rows of
// 64 bytes, 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3)): start
// address >> 4, leading byte offset 16 (unused by this layout), stride byte
// offset 512 (next group of 8 rows), version 1 at bit 46, layout type 4
// (SWIZZLE_64B) at bits 61-63.  K-step k of 32 e4m3 starts 32*k bytes in.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(512 >> 4) << 32) |
         (1ull << 46) | (4ull << 61);
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

// TMA loads of one tile, both completing on mbarrier bar: rows [y, y + 128)
// of the key tensor (all 64 bytes of each) into dst with the 64-byte
// swizzle, and scales [x, x + kScaleBox) into sdst.  Elements past the end of
// a tensor read as 0.
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap* keys, int32_t y,
                                              uint32_t sdst, const CUtensorMap* scales, int32_t x,
                                              uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"((uint32_t)(kRawBytes + 2 * kScaleBox))
               : "memory");
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2}], [%3];" ::"r"(sdst),
      "l"(reinterpret_cast<uint64_t>(scales)), "r"(x), "r"(bar)
      : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(keys)), "r"(0), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (tensor memory) [+]= A (shared) . B (shared)^T, e4m3 x e4m3 -> f32
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %4, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(accumulate), "r"(kIdesc)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// This thread's tensor-memory lane, 16 / 8 consecutive 32-bit columns.  The
// registers are valid only after tc_wait_ld(); tc_reg_fence() after the wait
// keeps the compiler from reading them earlier.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
#if QSA_K1_PIECES != 6
__device__ __forceinline__ void tc_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
#endif
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void tc_reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// e4m3 code (round to nearest even, saturating at +-448) of x, and its value.
__device__ __forceinline__ uint8_t to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_value(uint8_t c) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ int unit_of_tile(const IndexScoreParams& p, int t) {
  int lo = 0, hi = p.b.n_units - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Work counters: the workspace keeps two int32 per request x layer.  The
// first of unit u counts the unit's tiles handed out; the second of the
// call's first unit counts the CTAs that have finished.
__device__ __forceinline__ int32_t* unit_counter(const BatchDesc& b, int u) {
  return b.tickets + 2 * ((int64_t)b.u[u].req * b.n_layers + b.u[u].layer);
}

__device__ __forceinline__ int ld_relaxed_gpu(const int32_t* ptr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// Write unit u's query pieces into the B slot at B (whole warp) and return the
// exponent s of the common scale 2^s (so that max |q| * 2^s is in [128, 256)).
__device__ __forceinline__ int build_pieces(const IndexScoreParams& p, int u, uint8_t* B, int lane) {
  const float* qu = p.q_idx + (int64_t)u * kIndexHeads * kIndexDim;
  constexpr int kPerLane = kIndexHeads * kIndexDim / 32;   // 16
  float qv[kPerLane];
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < kPerLane; ++k) {
    qv[k] = qu[lane + 32 * k];
    m = fmaxf(m, fabsf(qv[k]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  int e = 0;
  if (m > 0.f) frexpf(m, &e);                // m = f * 2^e, f in [0.5, 1)
  int s = m > 0.f ? 8 - e : 0;
  s = s < -126 ? -126 : (s > 126 ? 126 : s);   // 2^s a normal fp32
  const float two_s = __int_as_float((127 + s) << 23);
  // zero the padding rows kPieces*8 .. kN-1 (whole 16-byte chunks)
  for (int c = lane; c < (kN - kPieces * kIndexHeads) * kIndexDim / 16; c += 32)
    *reinterpret_cast<uint4*>(B + kPieces * kIndexHeads * kIndexDim + 16 * c) = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int k = 0; k < kPerLane; ++k) {
    const int el = lane + 32 * k, h = el >> 6, d = el & 63;
    float r = qv[k] * two_s;                 // exact
#pragma unroll
    for (int pc = 0; pc < kPieces; ++pc) {
      const uint8_t c = to_e4m3(r);
      r = (r - e4m3_value(c)) * 16.f;        // exact residual, scaled up for the next piece
      const int row = pc * kIndexHeads + h;
      // 64-byte swizzle: chunk (d >> 4) of row `row` at chunk (d >> 4) ^ ((row >> 1) & 3)
      B[row * kIndexDim + ((((d >> 4) ^ (row >> 1)) & 3) << 4) + (d & 15)] = c;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  return s;
}

__global__ void __maxnreg__(QSA_K1_MAXREG)
index_score_tc_kernel(const __grid_constant__ IndexScoreParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled stages and B slots need 1024-byte alignment
  uint8_t* smem0 = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pl = warp / kPipeWarps, role = warp % kPipeWarps;
  uint8_t* smem = smem0 + pl * kPipeBytes;          // this warp's pipeline
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + kOffBar;
  constexpr int kBarD = 2 * kStages, kBarB = kBarD + 2 * kDBufs, kBarDone = kBarB + 2 * kBSlots;
  auto full = [&](int i) { return bars + 8u * (uint32_t)i; };
  auto empty = [&](int i) { return bars + 8u * (uint32_t)(kStages + i); };
  auto d_full = [&](int i) { return bars + 8u * (uint32_t)(kBarD + i); };
  auto d_empty = [&](int i) { return bars + 8u * (uint32_t)(kBarD + kDBufs + i); };
  auto b_full = [&](int i) { return bars + 8u * (uint32_t)(kBarB + i); };
  auto b_empty = [&](int i) { return bars + 8u * (uint32_t)(kBarB + kBSlots + i); };
  const uint32_t mma_done = bars + 8u * (uint32_t)kBarDone;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem0 + kOffTmemSlot);
  int4* stage_meta = reinterpret_cast<int4*>(smem + kOffStageMeta);  // ordered by the mbarrier asm
  const int total = p.tile_start[p.b.n_units];

  if (warp == kRoleMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)), "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (role == kRoleProd && lane == 0) {
    // a stage is free again once its MMAs have read the codes (one commit)
    // and the 128 workers have read the metadata and scales
    for (int i = 0; i < kStages; ++i) { mbar_init(full(i), 1); mbar_init(empty(i), 129); }
    for (int i = 0; i < kDBufs; ++i) { mbar_init(d_full(i), 1); mbar_init(d_empty(i), 128); }
    for (int i = 0; i < kBSlots; ++i) { mbar_init(b_full(i), 1); mbar_init(b_empty(i), 1); }
    mbar_init(mma_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.keys_map)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.scales_map)) : "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot + (uint32_t)pl * kPipeCols;   // this pipeline's columns
  // Everything above touches only shared and tensor memory and the
  // parameters, so it overlaps the tail of the kernel before this one;
  // the work counters, the query and the keys are read only after it.
  grid_dependency_wait();

  if (role == kRoleProd) {
    // ---- producer (whole warp; lane 0 does the atomics, waits and copies).
    // Stream position i holds the i-th tile this pipeline takes; after the
    // last one the producer marks the end in the next position.
    // Work: chunks of kChunk tiles of one unit from that unit's counter.  A
    // pipeline starts on its home unit (pipelines spread over the units in
    // proportion to their tiles) and stays on a unit until it runs dry, then
    // moves to the unit with the most tiles left; so it switches units (and
    // builds query pieces) rarely.  The next chunk is taken one chunk early.
    const int n_units = p.b.n_units;
    const int n_pipes = (int)gridDim.x * kPipes, me = (int)blockIdx.x * kPipes + pl;
    auto tiles_of = [&](int v) { return p.tile_start[v + 1] - p.tile_start[v]; };
    int cu = unit_of_tile(p, (int)((int64_t)me * total / n_pipes));
    int c0 = 0, c1 = 0;               // current chunk: local tiles [c0, c1) of unit cu
    int pre = 0;                      // next chunk of unit cu (lane 0), valid when have_pre
    bool have_pre = false, first = true;
    int i = 0, run = -1, run_u = -1, s_run = 0;
    int64_t row0 = p.b.unit_row(cu);
    bool ok = true;
    for (;;) {
      // ---- next chunk
      bool done = false;
      for (;;) {
        if (have_pre) {
          have_pre = false;
          const int t = __shfl_sync(0xFFFFFFFFu, pre, 0);
          if (t < tiles_of(cu)) { c0 = t; break; }
        }
        int uu = cu;
        if (!first) {
          // the unit with the most tiles left (lowest index on ties)
          int rem = 0;
          uu = -1;
          for (int v = lane; v < n_units; v += 32) {
            const int rv = tiles_of(v) - ld_relaxed_gpu(unit_counter(p.b, v));
            if (rv > rem) { rem = rv; uu = v; }
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
        int t = 0;
        if (lane == 0) t = atomicAdd(unit_counter(p.b, uu), kChunk);
        t = __shfl_sync(0xFFFFFFFFu, t, 0);
        if (t < tiles_of(uu)) {
          if (uu != cu) { cu = uu; row0 = p.b.unit_row(cu); }
          c0 = t;
          break;
        }
      }
      if (done) break;
      c1 = c0 + kChunk < tiles_of(cu) ? c0 + kChunk : tiles_of(cu);
      if (c1 < tiles_of(cu)) {          // take the next chunk of this unit early
        if (lane == 0) pre = atomicAdd(unit_counter(p.b, cu), kChunk);
        have_pre = true;
      }
      if (cu != run_u) {
        // new run: pieces of unit cu into slot run & 1, once the MMAs of
        // run - 2 (the slot's last user) have completed
        ++run;
        const int slot = run & 1;
        if (run >= 2) {
          if (lane == 0) ok = mbar_wait(b_empty(slot), (uint32_t)((run >> 1) - 1) & 1u, p.b.err, run);
          ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
          if (!ok) break;
        }
        s_run = build_pieces(p, cu, smem + kOffB + slot * kBBytes, lane);
        run_u = cu;
        if (lane == 0) mbar_arrive(b_full(slot));
      }
      if (lane == 0) {
        for (int t = c0; t < c1; ++t, ++i) {
          const int st = i % kStages;
          if (i >= kStages && !(ok = mbar_wait(empty(st), (uint32_t)(i / kStages - 1) & 1u, p.b.err, t)))
            break;
          const int64_t row = row0 + (int64_t)t * kTile;   // first row of the tile
          const int64_t x0 = row & ~7ll;
          stage_meta[st] = make_int4(cu, t, run | ((s_run + 1024) << kRunBits), (int)(row - x0));
          tma_load_tile(sb + kOffRaw + st * kRawBytes, &p.keys_map, (int32_t)row,
                        sb + kOffScale + st * kScaleSlot, &p.scales_map, (int32_t)x0, full(st));
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      i = __shfl_sync(0xFFFFFFFFu, i, 0);
      if (!ok) break;
    }
    if (lane == 0) {
      // no copy of this pipeline may still be landing when the CTA exits:
      // wait for the last load of every stage (on the normal path the
      // consumers do too)
      for (int j = (i > kStages ? i - kStages : 0); j < i && ok; ++j)
        ok = mbar_wait(full(j % kStages), (uint32_t)(j / kStages) & 1u, p.b.err, -1);
      // end marker (the MMA lane and the workers read it)
      const int st = i % kStages;
      if (ok && (i < kStages || mbar_wait(empty(st), (uint32_t)(i / kStages - 1) & 1u, p.b.err, -1))) {
        stage_meta[st] = make_int4(kEndOfWork, 0, 0, 0);
        mbar_arrive(full(st));
      }
    }
  } else if (role == kRoleMma) {
    // ---- MMA issue, lane 0 alone: per tile two tcgen05.mma (K = 32 each)
    // into one accumulator, then commits that free the stage and publish the
    // accumulator.  At a new run the lane releases the previous run's B slot
    // (commit: arrives once those MMAs are done) and waits for the new slot.
    if (lane == 0) {
      int cur_run = -1;
      for (int i = 0;; ++i) {
        const int st = i % kStages, db = i % kDBufs;
        if (!mbar_wait(full(st), (uint32_t)(i / kStages) & 1u, p.b.err, i)) break;
        const int4 m = stage_meta[st];
        if (m.x < 0) break;
        const int run = m.z & ((1 << kRunBits) - 1);
        if (run != cur_run) {
          if (cur_run >= 0) tc_commit(b_empty(cur_run & 1));
          cur_run = run;
          if (!mbar_wait(b_full(run & 1), (uint32_t)(run >> 1) & 1u, p.b.err, run)) break;
        }
        if (i >= kDBufs && !mbar_wait(d_empty(db), (uint32_t)(i / kDBufs - 1) & 1u, p.b.err, i)) break;
        tc_fence_after();
        const uint32_t a0 = sb + kOffRaw + st * kRawBytes;
        const uint32_t b0 = sb + kOffB + (run & 1) * kBBytes;
        const uint32_t d = tmem + (uint32_t)(db * kDStride);
        tc_mma_f8(d, smem_desc_sw64(a0), smem_desc_sw64(b0), 0u);
        tc_mma_f8(d, smem_desc_sw64(a0 + 32), smem_desc_sw64(b0 + 32), 1u);
        tc_commit(empty(st));
        tc_commit(d_full(db));
      }
      // every MMA issued above has completed once this arrives
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, p.b.err, -1);
    }
    __syncwarp();
  } else {
    // ---- workers: thread = token row r of the tile = tensor-memory lane r
    // (lane quarter warp % 4).
    const int qtr = warp & 3;
    const int r = qtr * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qtr * 32) << 16);
    int eu = -1;                       // unit of the scoring cursor
    int64_t en = 0;
    float* out = nullptr;
    float wr[kIndexHeads];             // the unit's head weights
#pragma unroll
    for (int h = 0; h < kIndexHeads; ++h) wr[h] = 0.f;
    for (int i = 0;; ++i) {
      const int st = i % kStages, db = i % kDBufs;
      if (!mbar_wait(full(st), (uint32_t)(i / kStages) & 1u, p.b.err, i)) break;
      const int4 m = stage_meta[st];
      if (m.x < 0) break;
      const float sc_raw = __half2float(__ushort_as_half(
          *reinterpret_cast<const uint16_t*>(smem + kOffScale + st * kScaleSlot + 2 * (m.w + r))));
      mbar_arrive(empty(st));
      // undo the pieces' common scale 2^s together with the token's scale
      const float sc = ldexpf(sc_raw, -((m.z >> kRunBits) - 1024));
      if (m.x != eu) {
        eu = m.x;
        en = p.b.u[eu].n;
        out = p.blk + (int64_t)eu * p.blk_stride;
#pragma unroll
        for (int h = 0; h < kIndexHeads; ++h) wr[h] = __ldg(p.w + (int64_t)eu * kIndexHeads + h);
      }
      if (!mbar_wait(d_full(db), (uint32_t)(i / kDBufs) & 1u, p.b.err, i)) break;
      tc_fence_after();
      // columns 8p + h: piece p of head h; y_h = sum_p 16^-p * D[8p + h] (Horner)
      const uint32_t dcol = lane_base + (uint32_t)(db * kDStride);
      float y[kIndexHeads];
      {
        auto f = [](uint32_t x) { return __uint_as_float(x); };
#if QSA_K1_PIECES == 6
        uint32_t v45[16], v23[16], v01[16];
        tc_ld16(dcol + 32, v45);
#else
        uint32_t v4[8], v23[16], v01[16];
        tc_ld8(dcol + 32, v4);
#endif
        tc_ld16(dcol + 16, v23);
        tc_ld16(dcol, v01);
        tc_wait_ld();
#if QSA_K1_PIECES == 6
        tc_reg_fence(v45);
#else
        tc_reg_fence(v4);
#endif
        tc_reg_fence(v23);
        tc_reg_fence(v01);
#pragma unroll
        for (int h = 0; h < kIndexHeads; ++h) {
#if QSA_K1_PIECES == 6
          float a = fmaf(f(v45[8 + h]), 0.0625f, f(v45[h]));
          a = fmaf(a, 0.0625f, f(v23[8 + h]));
#else
          float a = fmaf(f(v4[h]), 0.0625f, f(v23[8 + h]));
#endif
          a = fmaf(a, 0.0625f, f(v23[h]));
          a = fmaf(a, 0.0625f, f(v01[8 + h]));
          y[h] = fmaf(a, 0.0625f, f(v01[h]));
        }
      }
      tc_fence_before();
      mbar_arrive(d_empty(db));
      const int64_t tok = (int64_t)m.y * kTile + r;
      float s = -INFINITY;
      if (tok < en) {
        s = 0.f;
#pragma unroll
        for (int h = 0; h < kIndexHeads; ++h) s = fmaf(wr[h], fmaxf(y[h] * sc, 0.f), s);
      }
      s = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
      s = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
      if ((lane & 3) == 0 && tok < en) out[tok >> 2] = s;
    }
  }

  tc_fence_before();
  __syncthreads();
  trigger_dependents();
  tc_fence_after();
  if (warp == kRoleMma)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tmem_slot),
                 "r"(kTmemCols)
                 : "memory");
  // the last CTA to finish re-arms the work counters for the next call
  if (tid == 0) {
    int32_t* finished = unit_counter(p.b, 0) + 1;
    __threadfence();
    if (atomicAdd(finished, 1) == (int)gridDim.x - 1) {
      __threadfence();
      for (int uu = 0; uu < p.b.n_units; ++uu)
        *reinterpret_cast<volatile int32_t*>(unit_counter(p.b, uu)) = 0;
      *reinterpret_cast<volatile int32_t*>(finished) = 0;
    }
  }
}

}  // namespace

cudaError_t make_index_maps(CUtensorMap* keys_map, const void* keys, CUtensorMap* scales_map,
                            const void* scales, int64_t rows) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);
  static const Encode encode = [] {   // resolved once, thread-safe
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                           cudaEnableDefault, &q);
    return (e == cudaSuccess && q == cudaDriverEntryPointSuccess) ? reinterpret_cast<Encode>(fn)
                                                                   : nullptr;
  }();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)kIndexDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kIndexDim};
  const cuuint32_t box[2] = {(cuuint32_t)kIndexDim, (cuuint32_t)kTile};
  const cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = encode(keys_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(keys), dims,
                      strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const cuuint64_t sdims[1] = {(cuuint64_t)rows};
  const cuuint32_t sbox[1] = {(cuuint32_t)kScaleBox};
  r = encode(scales_map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 1, const_cast<void*>(scales), sdims,
             strides /* unused at rank 1 */, sbox, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_index_score(const BatchDesc& b, const CUtensorMap* keys_map,
                               const CUtensorMap* scales_map, const float* q_idx, const float* w,
                               float* blk_scores, int64_t blk_stride, cudaStream_t s) {
  static PerDeviceOnce setup;
  cudaError_t e = setup.run([] { return prefer_max_shared(index_score_tc_kernel, kSmemBytes); });
  int sm_count = 0;
  if (e == cudaSuccess) e = current_sm_count(&sm_count);
  if (e != cudaSuccess) return e;
  IndexScoreParams p;
  p.keys_map = *keys_map;
  p.scales_map = *scales_map;
  p.b = b;
  p.q_idx = q_idx;
  p.w = w;
  p.blk = blk_scores;
  p.blk_stride = blk_stride;
  int64_t tiles = 0;
  for (int u = 0; u < b.n_units; ++u) {
    p.tile_start[u] = (int32_t)tiles;
    tiles += (b.u[u].n + kTile - 1) / kTile;
  }
  p.tile_start[b.n_units] = (int32_t)tiles;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > (1ll << 30)) return cudaErrorInvalidValue;
  const int64_t cap = (int64_t)kCtasPerSm * sm_count;
  const int64_t chunks = (tiles + kChunk - 1) / kChunk;
  const unsigned grid = (unsigned)(chunks < cap ? chunks : cap);
  return launch_kernel(index_score_tc_kernel, dim3(grid), dim3(kThreadsTc), kSmemBytes, s, 0, dim3(1), p);
}

}  // namespace qsa
