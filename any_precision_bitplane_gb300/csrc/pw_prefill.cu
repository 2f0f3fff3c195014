// Fused mixed-precision MoE layer, prefill path (many tokens per expert).
//
// PagedWeight, "Core components" 3 (fused mixed-precision kernel): every
// block is read from its top q_i bitplanes and LUT at its own bitwidth.  With
// hundreds of tokens per expert the layer is a dense contraction, so this path
// dequantises weight tiles into shared memory and runs them through the
// tensor cores:
//
//   permute    pairs grouped by expert (offsets, perm)          [pw_route.cu]
//   gather     xg[pos] = fp16(hidden[perm[pos] / k] * 2^-e_pos), with the
//              power of two that puts the row's largest magnitude in [1, 2)
//              (stored as scale[pos] = 2^e_pos)           (one warp per row)
//   gate_up    per (expert, 64 gate/up row pairs, 512 tokens):  D = W_gu x^T
//              in TMEM, epilogue g, u = D * 2^e, h = SiLU(g) * u ->
//              fp16 h[pos] * 2^-2e, computed as Dg * Du * sigma(Dg * 2^e)
//   down       per (expert, 128 down rows, 512 tokens, K half): D = W_dn h^T
//              over one half of K, epilogue y = D * 2^2e -> y[pair] or
//              y2[pair] (fp32)
// The row scales keep every fp16 operand in range for any finite input:
// |x * 2^-e| < 2, and h * 2^-2e is about (g 2^-e)(u 2^-e), bounded by the
// weights.
//   combine    out[t] = sum_j w_tj * (y + y2)[t*k + j], j order (one pass)
//
// GEMM kernel: one CTA per SM, persistent, 27 warps in five roles.
//   warp 20     scheduler and token-operand producer: takes tile ids from a
//               global counter (SMs that draw cheap tiles take more of them),
//               publishes each through a 4-deep ring in shared memory, and
//               TMA-loads the fp16 token rows (64-byte swizzle) of every k-step.
//   warp 21     plane producer: per k-step (32 columns = one plane word
//               column), copies the words of the tile's 128 rows from each
//               of the top q planes into a 6-deep ring (a word column of
//               consecutive rows is contiguous: two 256-byte runs for a
//               gate_up tile, one 512-byte run for a down tile) with 16-byte
//               cp.async per lane, whose completion arrives on the stage's
//               barrier; the copy engine stays free for the token operand.
//   warps 0-15  dequant: two sets of eight that take alternate k-steps.  In a
//               set, four warps own columns 0-15 of the k-step and four own
//               columns 16-31; each thread owns one A row.  A thread reads
//               its row's q plane words from the ring, rebuilds 16 indices
//               with a byte transpose and an 8x8 bit-matrix transpose, looks
//               them up in the row's LUT (fp16, shared memory, every lane of
//               a warp on its own bank) and writes 32 bytes of the
//               64-byte-swizzled, K-major A stage.
//   warp 22     allocates the 512 TMEM columns; lane 0 issues per k-step two
//               K=16 steps of two tcgen05.mma (M=128, N=256 each, fp16 x
//               fp16 -> fp32) into columns [0,256) and [256,512), with one
//               wait per stage: a stage's A rows and token rows complete one
//               barrier.
//   warps 16-19 and 23-26: epilogue, two groups of four (TMEM lane quarter =
//               warp % 4) that take alternate 32-column chunks of the
//               accumulator, so that it is drained twice as fast (the MMA
//               waits for the drained accumulator before the next tile).
//               gate_up: gate and up rows of one h column sit 8 lanes apart,
//               so one lane exchange pairs them; h = SiLU(g) * u (fp16) is
//               staged in shared memory (one buffer per group) and written
//               out as 128-byte rows.  down: y rows (fp32) go straight to
//               each pair's output row.
// A weight tile is dequantised once per 512 tokens.  Stages are handed over
// with mbarriers; every wait is bounded, and a timeout latches PW_ERR_TIMEOUT
// and unwinds without trapping.  Decisions that named barriers depend on are
// taken by one thread and shared through shared memory, so every thread of a
// barrier group takes the same path even while unwinding.
//
// Operand precision: the weights are exact fp16 LUT values; hidden states are
// scaled by a power of two per row and converted bf16 -> fp16 (exact unless a
// value falls below fp16's normal range relative to its row's largest, i.e.
// below 2^-14 of it); h is stored as fp16 (scaled); all accumulation is fp32.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "pw_bits.cuh"
#include "pw_internal.cuh"

namespace pw {
namespace {

constexpr int BM = 128;                 // A rows per tile (MMA M)
constexpr int BN = 512;                 // tokens per tile: two MMAs of N = 256
constexpr int BNH = 256;                // tokens per MMA
constexpr int BK = 32;                  // K per stage: one plane word column, 64-byte rows
constexpr int NST = 3;                  // A/B pipeline stages
constexpr int NPS = 6;                  // plane-word stages
constexpr int kDqWarps = 16;            // warps 0-15
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kSetThreads = kDqThreads / 2;
constexpr int kEpiWarp0 = 16;           // warps 16-19: epilogue group 0
constexpr int kSchedWarp = 20;
constexpr int kPlaneWarp = 21;
constexpr int kMmaWarp = 22;
constexpr int kEpiWarp1 = 23;           // warps 23-26: epilogue group 1
constexpr int kEpiThreads = 256;        // both groups
constexpr int kThreads = 27 * 32;
constexpr int kTileRing = 4;
constexpr int kTileConsumers = 4;       // dequant, epilogue, plane producer, MMA issuer
constexpr uint32_t kAStage = BM * BK * 2;     // 8 KB
constexpr uint32_t kBHalf = BNH * BK * 2;     // 16 KB per 256 tokens
constexpr uint32_t kBStage = 2 * kBHalf;      // 32 KB
constexpr uint32_t kPlaneStage = 8 * BM * 4;  // up to 8 planes x 128 words
constexpr uint32_t kLutBytes = 256 * BM * 2;  // fp16 [256][128]
constexpr uint32_t kStageBuf = 32 * 64 * 2;   // epilogue: 32 tokens x 64 h columns, fp16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSpinLimit = 1u << 24;
constexpr int kMaxExperts = 1024;

// Shared memory (offsets from the dynamic base, which must be 1024-aligned):
// the LUT sits at offset 0 so that lookups address the dynamic symbol with a
// register offset only; the plane-word ring, the epilogue buffers, barriers
// and tile prefix follow; the A/B stages come last.
constexpr uint32_t kOffLut = 0;
constexpr uint32_t kOffPlanes = kOffLut + kLutBytes;
constexpr uint32_t kOffStage = kOffPlanes + NPS * kPlaneStage;
constexpr uint32_t kOffBar = kOffStage + 2 * kStageBuf;        // 8-byte barriers
// kBarFull[i]: stage i holds its A rows (dequant arrivals) and its token rows
// (the token producer's arrival with the expected bytes, and the copies).
constexpr int kBarFull = 0, kBarEmpty = NST, kBarPlFull = 2 * NST,
              kBarPlEmpty = 2 * NST + NPS, kBarTileFull = 2 * NST + 2 * NPS,
              kBarTileEmpty = kBarTileFull + kTileRing, kBarAccFull = kBarTileEmpty + kTileRing,
              kBarAccEmpty = kBarAccFull + 1, kBarFinal = kBarAccEmpty + 1,
              kNumBars = kBarFinal + 1;
// misc words: [0] TMEM base, [1] abort flag, [2..5] tile ring, [6..7] dequant
// tile slots, [8..9] epilogue tile slots, [10] epilogue accumulator flag
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;
constexpr uint32_t kOffPrefix = kOffMisc + 64;                 // tile prefix [E+1]
constexpr uint32_t kOffA = (kOffPrefix + 4 * (kMaxExperts + 1) + 1023) & ~1023u;
constexpr uint32_t kOffB = kOffA + NST * kAStage;
constexpr size_t kSmemBytes = kOffB + NST * kBStage;
static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");
static_assert(kOffB % 1024 == 0 && kOffA % 1024 == 0, "swizzled stages need 1024-byte alignment");

extern __shared__ __align__(1024) unsigned char g_psmem[];

// ---------------------------------------------------------------- trace
//
// Built with -DPW_TRACE (build.py --trace, a separate library), the gate_up
// GEMM records %globaltimer stamps (ns) of every kTraceStride-th CTA (up to
// kTraceCtas of them) into a device buffer that pw_debug_gemm_trace copies
// out: per k-step of the CTA's first kTraceSteps (its ring position), when the
// MMA issuer found the stage full and when it had issued it, when a dequant
// set had written it and when the token producer found it empty; per tile
// (first kTraceTiles), the MMA start (accumulator free) and end (last
// commit), the epilogue's start and end and the dequant warps' LUT load; and
// the SM each traced CTA ran on.  The launch path clears the record before
// each gate_up launch.  Without PW_TRACE every hook is empty.
constexpr int kTraceSteps = 256, kTraceTiles = 32, kTraceCtas = 16;
struct GemmTrace {
  unsigned long long step[kTraceCtas][kTraceSteps][4];   // ready, issued, dequantised, empty seen
  // per k-step and dequant warp of its set (8): the warp's wait for the
  // stage's release done, its announcement of the stage's A rows done, its
  // wait for the plane words done, its index transpose done
  unsigned long long dq[kTraceCtas][kTraceSteps][8][4];
  unsigned long long tile[kTraceCtas][kTraceTiles][6];   // mma start, mma end, epi start, epi end,
                                                         // lut start, lut end
  unsigned long long smid[kTraceCtas];                   // SM id + 1 (0: CTA not traced)
};
#ifdef PW_TRACE
constexpr int kTraceStride = 10;
__device__ GemmTrace g_trace;
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int trace_slot() {
  const int b = static_cast<int>(blockIdx.x);
  return (b % kTraceStride == 0 && b / kTraceStride < kTraceCtas) ? b / kTraceStride : -1;
}
#define PW_TRACE_STEP(mode, i, k)                                                           \
  do {                                                                                      \
    const int ts_ = trace_slot();                                                           \
    if ((mode) == kGateUp && ts_ >= 0 && (i) < static_cast<uint32_t>(kTraceSteps))           \
      g_trace.step[ts_][(i)][(k)] = trace_now();                                            \
  } while (0)
#define PW_TRACE_TILE(mode, j, k)                                                           \
  do {                                                                                      \
    const int ts_ = trace_slot();                                                           \
    if ((mode) == kGateUp && ts_ >= 0 && (j) < static_cast<uint32_t>(kTraceTiles))           \
      g_trace.tile[ts_][(j)][(k)] = trace_now();                                            \
  } while (0)
#define PW_TRACE_DQ(mode, i, k)                                                             \
  do {                                                                                      \
    const int ts_ = trace_slot();                                                           \
    if ((mode) == kGateUp && ts_ >= 0 && (i) < static_cast<uint32_t>(kTraceSteps) &&         \
        (threadIdx.x & 31) == 0)                                                            \
      g_trace.dq[ts_][(i)][(threadIdx.x >> 5) & 7][(k)] = trace_now();                      \
  } while (0)
__device__ __forceinline__ unsigned long long trace_now_after(uint32_t dep) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t) : "r"(dep));   // waits for dep
  return t;
}
#define PW_TRACE_DQ_AFTER(mode, i, k, dep)                                                  \
  do {                                                                                      \
    const int ts_ = trace_slot();                                                           \
    if ((mode) == kGateUp && ts_ >= 0 && (i) < static_cast<uint32_t>(kTraceSteps) &&         \
        (threadIdx.x & 31) == 0)                                                            \
      g_trace.dq[ts_][(i)][(threadIdx.x >> 5) & 7][(k)] = trace_now_after(dep);             \
  } while (0)
#define PW_TRACE_SM(mode)                                                                   \
  do {                                                                                      \
    const int ts_ = trace_slot();                                                           \
    if ((mode) == kGateUp && ts_ >= 0 && threadIdx.x == 0) {                                \
      unsigned sm_;                                                                         \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                                      \
      g_trace.smid[ts_] = sm_ + 1ull;                                                       \
    }                                                                                       \
  } while (0)
#else
#define PW_TRACE_STEP(mode, i, k) do { } while (0)
#define PW_TRACE_TILE(mode, j, k) do { } while (0)
#define PW_TRACE_SM(mode) do { } while (0)
#define PW_TRACE_DQ(mode, i, k) do { } while (0)
#define PW_TRACE_DQ_AFTER(mode, i, k, dep) do { } while (0)
#endif

enum Mode { kGateUp = 0, kDown = 1 };

struct GemmArgs {
  int32_t H, I, E, k, n_pairs;
  const pw_block_entry* table;
  const int32_t* offsets;   // [E+1]
  const int32_t* perm;      // [n_pairs]
  const float* xscale;      // [n_pairs] 2^e of each grouped position's row
  __half* h_ws;             // [n_pairs][I] (gate_up writes, down reads through TMA)
  float* y_ws;              // [n_pairs][H]
  float* y_ws2;             // [n_pairs][H]: the second K half's partial sums (ksplit 2)
  int32_t ksplit;           // 1, or 2: each weight tile's K is split over two tiles
  int32_t* tile_counter;    // zeroed by the gather launch
  int32_t min_tokens;       // experts with fewer pairs get no tiles
  int32_t* status;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false if the CTA is aborting or the limit ran out (which
// latches the timeout and starts the abort).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int32_t* status, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  latch_status(status, PW_ERR_TIMEOUT);
  return false;
}

// Failure-detection check: the tensor-core kernels' bounded mbarrier wait,
// run by one thread on a barrier that expects one arrival that never comes
// (phase 0 never completes), with `limit` polls.  It must give up, latch
// PW_ERR_TIMEOUT, raise the abort flag and return.
__global__ void mbar_wait_check_kernel(int32_t* status, uint32_t limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit);
  }
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void named_sync_dq() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDqThreads) : "memory");
}

// K-major operand, 64-byte swizzle: rows of 64 bytes, 8-row atoms of 512
// bytes (stride-dimension offset), leading-dimension offset unused (1).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(512 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(4) << 61;
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B, both
// K-major, M = BM, N = n (a multiple of 16, at most 256).
__device__ __forceinline__ uint32_t make_idesc(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
}

// One k-step (K = 32: two K = 16 steps) of a tile: the MMAs of token half 0
// (A x B0 into columns [0, 256)) and, when `two`, of half 1 (A x B1 into
// [256, 512)), accumulating unless `first`, then their commit to `empty`, in
// one instruction block.
__device__ __forceinline__ void issue_kstep(uint32_t tmem, uint64_t a0, uint64_t a1, uint64_t b0,
                                            uint64_t b1, uint64_t c0, uint64_t c1, uint32_t id0,
                                            uint32_t id1, bool first, bool two, uint32_t empty) {
  asm volatile(
      "{\n\t.reg .pred pacc, ptwo, pone;\n\t"
      "setp.eq.b32 pacc, %10, 0;\n\t"
      "setp.ne.b32 ptwo, %11, 0;\n\t"
      "setp.eq.b32 pone, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %4, %8, pacc;\n\t"
      "@ptwo tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %6, %9, pacc;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %5, %8, pone;\n\t"
      "@ptwo tcgen05.mma.cta_group::1.kind::f16 [%1], %3, %7, %9, pone;\n\t"
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%12];\n\t}"
      ::"r"(tmem), "r"(tmem + BNH), "l"(a0), "l"(a1), "l"(b0), "l"(b1), "l"(c0), "l"(c1),
        "r"(id0), "r"(id1), "r"(static_cast<uint32_t>(first)), "r"(static_cast<uint32_t>(two)),
        "r"(empty)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// A 16-column TMEM load (32 lanes x 16 columns of 32 bits), issued without
// waiting: the registers are written when the load completes.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Waits for the thread's TMEM loads; naming the registers of the last load as
// operands keeps every use of them below the wait.
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Both epilogue groups (tile ids and the accumulator flag).
__device__ __forceinline__ void named_sync_epi() {
  asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory");
}

// One epilogue group (its staging buffer): barrier 3 or 4.
__device__ __forceinline__ void named_sync_epi_group(int group) {
  if (group)
    asm volatile("bar.sync 4, 128;" ::: "memory");
  else
    asm volatile("bar.sync 3, 128;" ::: "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The barrier receives one arrival when all of this thread's earlier
// cp.async copies have landed (its expected count includes that arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Wait for the completion of every phase of barriers [first, first + n) that
// the calling thread armed in its last `count` sequence numbers (so that
// copies still in flight land before the CTA unwinds).
__device__ void drain_copies(uint32_t bar_base, int first, int n, uint32_t seq_end,
                             uint32_t count) {
  for (uint32_t j = (seq_end > count ? seq_end - count : 0); j < seq_end; ++j) {
    const uint32_t bar = bar_base + 8 * (first + j % n);
    for (uint32_t i = 0; i < kSpinLimit && !mbar_try(bar, (j / n) & 1u); ++i) {
    }
  }
}

// ---------------------------------------------------------------- tile list

struct Tile {
  int e, m, n;  // expert, row tile, token tile
  int kh;       // K part (0, or 1 of 2 when the K range is split)
};

// The k-steps [k0, k0 + kc) of a tile: the whole K range, or one half of it.
struct KRange {
  int k0, kc;
};

__device__ __forceinline__ KRange k_range(const Tile& tile, int ksteps, int ksplit) {
  if (ksplit == 1) return KRange{0, ksteps};
  const int h = ksteps / 2;
  return tile.kh ? KRange{h, ksteps - h} : KRange{0, h};
}

__device__ __forceinline__ int m_tiles(Mode mode, const GemmArgs& a) {
  return mode == kGateUp ? a.I / 64 : a.H / BM;
}

// Tile t of the list ordered (expert, row tile, K part, token tile), token
// tile fastest (the token tiles of one weight tile run side by side, so the
// second read of its planes is an L2 hit).
__device__ __forceinline__ Tile tile_at(int t, const int* prefix, int E, const int32_t* offsets,
                                        int ksplit) {
  int lo = 0, hi = E;  // find e with prefix[e] <= t < prefix[e+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int local = t - prefix[e];
  const int nt = (offsets[e + 1] - offsets[e] + BN - 1) / BN;
  Tile r;
  r.e = e;
  r.n = local % nt;
  r.kh = (local / nt) % ksplit;
  r.m = local / (nt * ksplit);
  return r;
}

__device__ __forceinline__ bool tile_usable(Mode mode, const GemmArgs& a, int e) {
  const pw_block_entry gu = a.table[2 * e];
  if (gu.state != PW_PAGE_GPU || !supported_q(gu.q)) return false;
  if (mode == kDown) {
    const pw_block_entry dn = a.table[2 * e + 1];
    if (dn.state != PW_PAGE_GPU || !supported_q(dn.q)) return false;
  }
  return true;
}

// Latch why a tile of expert e cannot be computed (first error wins).
__device__ void report_unusable(Mode mode, const GemmArgs& a, int e) {
  const pw_block_entry ent = a.table[2 * e + (mode == kGateUp ? 0 : 1)];
  const pw_block_entry gu = a.table[2 * e];
  if (ent.state != PW_PAGE_GPU || gu.state != PW_PAGE_GPU)
    latch_status(a.status, PW_ERR_PAGE_NOT_RESIDENT);
  else
    latch_status(a.status, PW_ERR_UNSUPPORTED_Q);
}

// One consumer's next tile id from the scheduler's ring (single thread).
// INT_MAX once the CTA is unwinding.
__device__ __forceinline__ int ring_take(uint32_t bar_base, const volatile int* ring, uint32_t& seq,
                                         volatile int* abort, int32_t* status) {
  const uint32_t slot = seq % kTileRing, par = (seq / kTileRing) & 1u;
  ++seq;
  if (!mbar_wait(bar_base + 8 * (kBarTileFull + slot), par, abort, status)) return INT_MAX;
  const int t = ring[slot];
  mbar_arrive(bar_base + 8 * (kBarTileEmpty + slot));
  return t;
}

// ---------------------------------------------------------------- dequant

// Which A row, plane word and LUT slot a dequant thread owns.  Thread (w, L)
// (w = warp % 4, L = lane) reads word `word` of each plane in the stage, so a
// warp's reads are 32 consecutive words; its LUT slot puts lane L on bank L.
//   gate_up: A rows come in groups of 16: 8 gate rows, then the 8 up rows of
//            the same h columns; seg (0 gate, 1 up) = w / 2 and h column
//            hc = 32 (w % 2) + L of the tile's 64.
//   down:    A row 32 w + L.
struct DqRow {
  int r;          // A row (TMEM lane)
  int word;       // word index in a plane's 128-word stage slab
  int grow;       // row of the block
  uint32_t slot;  // byte offset of the row's entries in a 256-byte LUT line
};

__device__ __forceinline__ DqRow dq_row(Mode mode, const GemmArgs& a, int m, int w, int lane) {
  DqRow d;
  d.slot = static_cast<uint32_t>((w >> 1) * 128 + lane * 4 + (w & 1) * 2);
  if (mode == kGateUp) {
    const int seg = w >> 1, hc = 32 * (w & 1) + lane;
    d.word = seg * 64 + hc;
    d.r = 16 * (hc >> 3) + 8 * seg + (hc & 7);
    d.grow = seg * a.I + m * 64 + hc;
  } else {
    d.r = 32 * w + lane;
    d.word = d.r;
    d.grow = m * BM + d.r;
  }
  return d;
}

// The row's LUT into its slot: entry v at byte v*256 + slot (fp16).  The four
// threads that own a row (two sets x two column halves) each move a quarter.
template <int Q>
__device__ __forceinline__ void load_lut(const uint16_t* lut, int grow, uint32_t slot, int part) {
  constexpr int kEnt = 1 << Q;
  constexpr int kVec = kEnt / 8;
  constexpr int kPer = (kVec + 3) / 4;
  const uint4* src = reinterpret_cast<const uint4*>(lut + static_cast<long long>(grow) * kEnt);
  uint4 raw[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (part + 4 * i < kVec) raw[i] = __ldg(src + part + 4 * i);
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int vec = part + 4 * i;
    if (vec < kVec) {
      const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw[i]);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint16_t*>(g_psmem + kOffLut + (vec * 8 + j) * 256 + slot) = h[j];
    }
  }
}

// Q plane words (P[0] = most significant plane) -> the indices of 16 of the
// word's 32 columns, one per byte: `sel` picks bytes 0-1 (columns 0-15) or
// bytes 2-3 (columns 16-31).  Byte j of ib[m] is the index of column 4m + j
// of that half.
template <int Q>
__device__ __forceinline__ void planes_to_index_half(const uint32_t (&P)[Q], uint32_t sel,
                                                     uint32_t (&ib)[4], const BitConsts& bc) {
  uint32_t rr[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rr[i] = (i < Q) ? P[Q - 1 - i] : 0u;
  const uint32_t t0 = __byte_perm(rr[0], rr[1], sel), t2 = __byte_perm(rr[2], rr[3], sel);
  const uint32_t t4 = __byte_perm(rr[4], rr[5], sel), t6 = __byte_perm(rr[6], rr[7], sel);
  uint32_t lo0 = __byte_perm(t0, t2, 0x5410), hi0 = __byte_perm(t4, t6, 0x5410);
  uint32_t lo1 = __byte_perm(t0, t2, 0x7632), hi1 = __byte_perm(t4, t6, 0x7632);
  bit_transpose8(lo0, hi0, bc);
  bit_transpose8(lo1, hi1, bc);
  ib[0] = lo0;
  ib[1] = hi0;
  ib[2] = lo1;
  ib[3] = hi1;
}

// The fp16 weights of chunk cc (8 columns, 8cc .. 8cc + 7) of a row's
// 16-column half from the half's indices: entry v of the row's LUT at v * 256
// + slot (fp16).  packed[i] holds columns 8cc + 2i and 8cc + 2i + 1.
__device__ __forceinline__ void dequant_chunk(const uint32_t (&ib)[4], int cc, uint32_t slot,
                                              uint32_t (&packed)[4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t word = ib[2 * cc + h];
    uint32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t off = __byte_perm(word, slot, 0x6504 | (j << 4));
      v[j] = *reinterpret_cast<const uint16_t*>(g_psmem + off);
    }
    packed[2 * h] = __byte_perm(v[0], v[1], 0x5410);
    packed[2 * h + 1] = __byte_perm(v[2], v[3], 0x5410);
  }
}

// This thread's share of a tile's k-steps: set `set` takes k-steps set,
// set + 2, ...; `half` picks the 16 columns.
template <int Q>
__device__ void dequant_ksteps(const GemmArgs& a, Mode mode, const DqRow& d, int ksteps,
                               uint32_t it_base, int set, int half, uint32_t sbase,
                               uint32_t bar_base, volatile int* abort, const BitConsts& bc) {
  const uint32_t sel = half ? 0x7362u : 0x5140u;
  const uint32_t sw = (static_cast<uint32_t>(d.r) >> 1) & 3u;
  for (int ks = set; ks < ksteps; ks += 2) {
    const uint32_t it = it_base + ks;
    const uint32_t ps = it % NPS, pp = (it / NPS) & 1u;
    const uint32_t st = it % NST, sp = (it / NST) & 1u;
    if (!mbar_wait(bar_base + 8 * (kBarPlFull + ps), pp, abort, a.status)) break;
    PW_TRACE_DQ(mode, it, 2);
    const uint32_t pbase = kOffPlanes + ps * kPlaneStage + d.word * 4;
    uint32_t wd[Q];
#pragma unroll
    for (int p = 0; p < Q; ++p) wd[p] = *reinterpret_cast<const uint32_t*>(g_psmem + pbase + p * 512);
    mbar_arrive(bar_base + 8 * (kBarPlEmpty + ps));
    uint32_t ib[4];
    planes_to_index_half<Q>(wd, sel, ib, bc);
    PW_TRACE_DQ_AFTER(mode, it, 3, ib[0] ^ ib[1] ^ ib[2] ^ ib[3]);   // after the transpose
    if (!mbar_wait(bar_base + 8 * (kBarEmpty + st), sp ^ 1u, abort, a.status)) break;
    PW_TRACE_DQ(mode, it, 0);
    const uint32_t row_base = sbase + kOffA + st * kAStage + d.r * 64;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {   // 16-byte chunk 2*half + cc = 8 columns
      uint32_t packed[4];
      dequant_chunk(ib, cc, d.slot, packed);
      const uint32_t c = 2 * half + cc;
      const uint32_t dst = row_base + ((c ^ sw) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[0]),
                   "r"(packed[1]), "r"(packed[2]), "r"(packed[3])
                   : "memory");
    }
    fence_proxy_async();
    mbar_arrive(bar_base + 8 * (kBarFull + st));
    if ((threadIdx.x & 255) == 0) PW_TRACE_STEP(mode, it, 2);
    PW_TRACE_DQ(mode, it, 1);
  }
  (void)mode;
}

template <int Q>
__device__ __forceinline__ void dequant_tile(const GemmArgs& a, Mode mode, const pw_block_entry& ent,
                                             const DqRow& d, int ksteps, uint32_t it_base, int set,
                                             int half, uint32_t sbase, uint32_t bar_base,
                                             volatile int* abort, const BitConsts& bc) {
  if (threadIdx.x == 0) PW_TRACE_TILE(mode, it_base / ksteps, 4);
  load_lut<Q>(ent.lut, d.grow, d.slot, 2 * set + half);
  named_sync_dq();
  if (threadIdx.x == 0) PW_TRACE_TILE(mode, it_base / ksteps, 5);
  dequant_ksteps<Q>(a, mode, d, ksteps, it_base, set, half, sbase, bar_base, abort, bc);
}

// ---------------------------------------------------------------- epilogue

// gate_up: thread (quarter q, lane L) holds TMEM lane 32q + L.  Lanes L and
// L ^ 8 hold the gate and up rows of h column 16q + 8(L / 16) + L % 8; the
// gate lane finishes the even tokens, the up lane the odd ones.
__device__ void epilogue_gateup(const GemmArgs& a, const Tile& tile, int pos0, int ntok,
                                uint32_t tmem_base, int quarter, int lane, int group,
                                int tid_g, uint32_t sbase) {
  const int up = (lane >> 3) & 1;
  const int hc = 16 * quarter + 8 * (lane >> 4) + (lane & 7);
  const uint32_t buf = sbase + kOffStage + group * kStageBuf;
  const uint32_t lanes = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  // The group's chunks c = group, group + 2, ... (32 columns each) go in
  // halves of 16 columns; each half's TMEM load is issued before the previous
  // half is processed, and each chunk's scale load one chunk ahead.
  int c = group;
  if (c * 32 >= ntok) return;
  uint32_t ra[16], rb[16];
  tmem_ld16_issue(lanes + c * 32, ra);
  float sc_next = c * 32 + lane < ntok ? __ldg(a.xscale + pos0 + c * 32 + lane) : 1.f;
  tmem_wait16(ra);
  for (;;) {
    const float sc_l = sc_next;   // lane L: 2^e of the chunk's token L
    const int cn = c + 2;
    const bool more = cn < BN / 32 && cn * 32 < ntok;
    if (more) sc_next = cn * 32 + lane < ntok ? __ldg(a.xscale + pos0 + cn * 32 + lane) : 1.f;
    tmem_ld16_issue(lanes + c * 32 + 16, rb);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if (hf == 1) {
        tmem_wait16(rb);
        if (more) tmem_ld16_issue(lanes + cn * 32, ra);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const uint32_t w0 = hf ? rb[2 * jj] : ra[2 * jj];
        const uint32_t w1 = hf ? rb[2 * jj + 1] : ra[2 * jj + 1];
        const float v0 = __uint_as_float(w0), v1 = __uint_as_float(w1);
        const float send = up ? v0 : v1;
        const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
        const int tok = 2 * (8 * hf + jj) + up;
        const float sc = __shfl_sync(0xffffffffu, sc_l, tok);
        // with g = gs 2^e and u = us 2^e (gs, us: the accumulators of the
        // scaled operands), h 2^-2e = gs us sigma(g): one rescale, inside
        // sigma, and nothing that can overflow (sigma of a huge |g| is 0 or 1)
        const float gs = up ? recv : v0;
        const float us = up ? v1 : recv;
        const float sig = __fdividef(1.f, 1.f + __expf(-gs * sc));
        st_shared_u16(buf + (tok * 64 + hc) * 2, __half_as_ushort(__float2half_rn(gs * us * sig)));
      }
    }
    named_sync_epi_group(group);   // the chunk is staged
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int piece = tid_g + 128 * k2, tok = piece >> 3, part = piece & 7;
      const int n = c * 32 + tok;
      if (n < ntok) {
        uint4 val;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                     : "r"(buf + tok * 128 + part * 16));
        *reinterpret_cast<uint4*>(a.h_ws + static_cast<long long>(pos0 + n) * a.I + tile.m * 64 +
                                  part * 8) = val;
      }
    }
    named_sync_epi_group(group);   // the buffer is free for the group's next chunk
    if (!more) break;
    tmem_wait16(ra);
    c = cn;
  }
}

// down: thread (quarter q, lane L) holds row 128 m + 32 q + L of y; a warp's
// stores for one token are one 128-byte line.  Tiles of an expert that cannot
// be computed write zeros.
__device__ void epilogue_down(const GemmArgs& a, const Tile& tile, int pos0, int ntok, bool usable,
                              uint32_t tmem_base, int quarter, int lane, int group) {
  const int row = tile.m * BM + quarter * 32 + lane;
  float* const y = tile.kh ? a.y_ws2 : a.y_ws;   // each K part's partial sums
  for (int c = group; c < BN / 32; c += 2) {
    if (c * 32 >= ntok) break;
    // lane L holds the pair row and 2^e of the chunk's token L
    const int nl = c * 32 + lane;
    int pair_l = 0;
    float sc_l = 1.f;
    if (nl < ntok) {
      pair_l = __ldg(a.perm + pos0 + nl);
      sc_l = __ldg(a.xscale + pos0 + nl);
    }
    float v[32];
    if (usable) {
      tmem_ld32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + c * 32, v);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int pair = __shfl_sync(0xffffffffu, pair_l, j);
      const float sc = __shfl_sync(0xffffffffu, sc_l, j);
      // (v 2^e) 2^e: two steps, so that 2^2e itself never has to be finite
      if (c * 32 + j < ntok) y[static_cast<long long>(pair) * a.H + row] = v[j] * sc * sc;
    }
  }
}

// ---------------------------------------------------------------- the GEMM kernel

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    dq_gemm_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmap_b,
                   const BitConsts bc) {
  constexpr Mode mode = static_cast<Mode>(MODE);
  const uint32_t sbase = smem_u32(g_psmem);
  const uint32_t bar_base = sbase + kOffBar;
  uint32_t* misc = reinterpret_cast<uint32_t*>(g_psmem + kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* ring = reinterpret_cast<volatile int*>(misc + 2);
  volatile int* dq_slot = reinterpret_cast<volatile int*>(misc + 6);
  volatile int* epi_slot = reinterpret_cast<volatile int*>(misc + 8);
  int* prefix = reinterpret_cast<int*>(g_psmem + kOffPrefix);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = m_tiles(mode, a);
  const int K = (mode == kGateUp) ? a.H : a.I;
  const int ksteps = K / BK;
  // gate_up tiles always take the whole K range (a compile-time 1 here keeps
  // that instantiation free of the split's index arithmetic)
  const int ksplit = (mode == kGateUp) ? 1 : a.ksplit;
  PW_TRACE_SM(mode);
  if (sbase & 1023u) {   // the swizzled stages need a 1024-byte aligned base
    if (tid == 0) latch_status(a.status, PW_ERR_CUDA);
    return;
  }

  if (tid == 0) {
    *abort = 0;
    int run = 0;
    for (int e = 0; e < a.E; ++e) {
      prefix[e] = run;
      const int cnt = a.offsets[e + 1] - a.offsets[e];
      if (cnt >= a.min_tokens) run += mt * ksplit * ((cnt + BN - 1) / BN);
    }
    prefix[a.E] = run;
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar_base + 8 * (kBarFull + i), kSetThreads + 1);
      mbar_init(bar_base + 8 * (kBarEmpty + i), 1);
    }
    for (int i = 0; i < NPS; ++i) {
      mbar_init(bar_base + 8 * (kBarPlFull + i), 32);
      mbar_init(bar_base + 8 * (kBarPlEmpty + i), kSetThreads);
    }
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(bar_base + 8 * (kBarTileFull + i), 1);
      mbar_init(bar_base + 8 * (kBarTileEmpty + i), kTileConsumers);
    }
    mbar_init(bar_base + 8 * kBarAccFull, 1);
    mbar_init(bar_base + 8 * kBarAccEmpty, kEpiThreads);
    mbar_init(bar_base + 8 * kBarFinal, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(misc)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const int total = prefix[a.E];

  if (warp < kDqWarps) {
    // ---- dequant: set 0 = warps 0-7 (even k-steps), set 1 = warps 8-15
    const int set = warp >> 3, half = (warp >> 2) & 1, w = warp & 3;
    uint32_t it_base = 0, seq = 0, iter = 0;
    for (;; ++iter) {
      if (tid == 0) dq_slot[iter & 1] = ring_take(bar_base, ring, seq, abort, a.status);
      named_sync_dq();   // the previous tile's lookups are done; the tile id is visible
      const int t = dq_slot[iter & 1];
      if (t >= total) break;
      const Tile tile = tile_at(t, prefix, a.E, a.offsets, ksplit);
      if (!tile_usable(mode, a, tile.e)) continue;
      const pw_block_entry ent = a.table[2 * tile.e + (mode == kGateUp ? 0 : 1)];
      const DqRow d = dq_row(mode, a, tile.m, w, lane);
      const int kc = k_range(tile, ksteps, ksplit).kc;
      switch (ent.q) {
        case 3: dequant_tile<3>(a, mode, ent, d, kc, it_base, set, half, sbase, bar_base, abort, bc); break;
        case 4: dequant_tile<4>(a, mode, ent, d, kc, it_base, set, half, sbase, bar_base, abort, bc); break;
        case 5: dequant_tile<5>(a, mode, ent, d, kc, it_base, set, half, sbase, bar_base, abort, bc); break;
        case 6: dequant_tile<6>(a, mode, ent, d, kc, it_base, set, half, sbase, bar_base, abort, bc); break;
        default: dequant_tile<8>(a, mode, ent, d, kc, it_base, set, half, sbase, bar_base, abort, bc); break;
      }
      it_base += kc;
    }
  } else if (warp < kSchedWarp || warp >= kEpiWarp1) {
    // ---- epilogue: group 0 = warps 16-19, group 1 = warps 23-26
    const int group = warp >= kEpiWarp1 ? 1 : 0;
    const int quarter = warp & 3;
    const int tid_g = tid - (group ? kEpiWarp1 : kEpiWarp0) * 32;   // 0-127 in the group
    const int tid_e = tid_g + 128 * group;                           // 0-255
    volatile int* acc_ok = reinterpret_cast<volatile int*>(misc + 10);
    uint32_t acc_it = 0, seq = 0, iter = 0;
    for (;; ++iter) {
      if (tid_e == 0) epi_slot[iter & 1] = ring_take(bar_base, ring, seq, abort, a.status);
      named_sync_epi();
      const int t = epi_slot[iter & 1];
      if (t >= total) break;
      const Tile tile = tile_at(t, prefix, a.E, a.offsets, ksplit);
      const int pos0 = a.offsets[tile.e] + tile.n * BN;
      const int ntok = min(BN, a.offsets[tile.e + 1] - pos0);
      const bool usable = tile_usable(mode, a, tile.e);
      if (!usable) {
        if (tid_e == 0) report_unusable(mode, a, tile.e);
        if (mode == kDown) epilogue_down(a, tile, pos0, ntok, false, tmem_base, quarter, lane, group);
        continue;
      }
      if (tid_e == 0) {
        *acc_ok = mbar_wait(bar_base + 8 * kBarAccFull, acc_it & 1u, abort, a.status) ? 1 : 0;
        PW_TRACE_TILE(mode, acc_it, 2);
      }
      ++acc_it;
      named_sync_epi();
      if (!*acc_ok) break;
      tc_fence_after();
      if (mode == kGateUp)
        epilogue_gateup(a, tile, pos0, ntok, tmem_base, quarter, lane, group, tid_g, sbase);
      else
        epilogue_down(a, tile, pos0, ntok, true, tmem_base, quarter, lane, group);
      tc_fence_before();
      mbar_arrive(bar_base + 8 * kBarAccEmpty);
      if (tid_e == 0) PW_TRACE_TILE(mode, acc_it - 1, 3);
    }
  } else if (warp == kSchedWarp) {
    // ---- scheduler + TMA producer for the token operand
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
      uint32_t it = 0, seq = 0;
      for (;;) {
        const uint32_t slot = seq % kTileRing, par = (seq / kTileRing) & 1u;
        ++seq;
        if (!mbar_wait(bar_base + 8 * (kBarTileEmpty + slot), par ^ 1u, abort, a.status)) break;
        int t = atomicAdd(a.tile_counter, 1);
        if (t >= total) t = INT_MAX;
        ring[slot] = t;
        mbar_arrive(bar_base + 8 * (kBarTileFull + slot));
        if (t == INT_MAX) break;
        const Tile tile = tile_at(t, prefix, a.E, a.offsets, ksplit);
        if (!tile_usable(mode, a, tile.e)) continue;
        const int pos0 = a.offsets[tile.e] + tile.n * BN;
        const int ntok = min(BN, a.offsets[tile.e + 1] - pos0);
        const int halves = ntok > BNH ? 2 : 1;
        const KRange kr = k_range(tile, ksteps, ksplit);
        bool ok = true;
        for (int s = 0; s < kr.kc; ++s, ++it) {
          const uint32_t stage = it % NST, spar = (it / NST) & 1u;
          if (!mbar_wait(bar_base + 8 * (kBarEmpty + stage), spar ^ 1u, abort, a.status)) {
            ok = false;
            break;
          }
          PW_TRACE_STEP(mode, it, 3);
          const uint32_t full = bar_base + 8 * (kBarFull + stage);
          mbar_arrive_tx(full, halves * kBHalf);
          for (int h = 0; h < halves; ++h)
            tma_load_2d(sbase + kOffB + stage * kBStage + h * kBHalf, &tmap_b, (kr.k0 + s) * BK,
                        pos0 + h * BNH, full);
        }
        if (!ok) break;
      }
      if (*abort) drain_copies(bar_base, kBarFull, NST, it, NST);
    }
  } else if (warp == kPlaneWarp) {
    // ---- plane producer: lane 0 takes tiles and arms the stage barriers;
    // the copies of a k-step are issued by the lanes in parallel (one per
    // lane), which keeps the copy engine fed.
    {
      uint32_t pit = 0, seq = 0;
      const long long N = (mode == kGateUp) ? 2LL * a.I : a.H;
      const long long plane_stride = N * ksteps;
      for (;;) {
        int t0 = 0;
        if (lane == 0) t0 = ring_take(bar_base, ring, seq, abort, a.status);
        const int t = __shfl_sync(0xffffffffu, t0, 0);
        if (t >= total) break;
        const Tile tile = tile_at(t, prefix, a.E, a.offsets, ksplit);
        if (!tile_usable(mode, a, tile.e)) continue;
        const pw_block_entry ent = a.table[2 * tile.e + (mode == kGateUp ? 0 : 1)];
        const int q = ent.q;
        const uint32_t* base =
            ent.planes + ((mode == kGateUp) ? static_cast<long long>(tile.m) * 64
                                            : static_cast<long long>(tile.m) * BM);
        const KRange kr = k_range(tile, ksteps, ksplit);
        bool ok = true;
        for (int s = 0; s < kr.kc; ++s, ++pit) {
          const uint32_t ps = pit % NPS, pp = (pit / NPS) & 1u;
          int ok0 = 1;
          if (lane == 0) ok0 = mbar_wait(bar_base + 8 * (kBarPlEmpty + ps), pp ^ 1u, abort, a.status);
          if (!__shfl_sync(0xffffffffu, ok0, 0)) {
            ok = false;
            break;
          }
          const uint32_t full = bar_base + 8 * (kBarPlFull + ps);
          const uint32_t dst = sbase + kOffPlanes + ps * kPlaneStage + lane * 16;
          // lane L copies 16 bytes of each plane: words 4L..4L+3 of the
          // stage slab (gate_up: lanes 0-15 the gate run, 16-31 the up run)
          const uint32_t* src = base + static_cast<long long>(kr.k0 + s) * N +
                                ((mode == kGateUp) ? ((lane >> 4) * a.I + (lane & 15) * 4) : lane * 4);
          for (int p = 0; p < q; ++p) cp_async16(dst + p * 512, src + p * plane_stride);
          cp_async_arrive(full);
        }
        if (!ok) break;
      }
      asm volatile("cp.async.wait_all;" ::: "memory");   // nothing in flight at exit
    }
  } else {
    // ---- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0, seq = 0;
      bool issued = false;
      for (;;) {
        const int t = ring_take(bar_base, ring, seq, abort, a.status);
        if (t >= total) break;
        const Tile tile = tile_at(t, prefix, a.E, a.offsets, ksplit);
        if (!tile_usable(mode, a, tile.e)) continue;
        const int pos0 = a.offsets[tile.e] + tile.n * BN;
        const int ntok = min(BN, a.offsets[tile.e + 1] - pos0);
        const int n0 = min(BNH, (ntok + 15) & ~15);
        const int n1 = ntok > BNH ? ((ntok - BNH + 15) & ~15) : 0;
        const uint32_t id0 = make_idesc(n0), id1 = make_idesc(n1 > 0 ? n1 : 16);
        if (!mbar_wait(bar_base + 8 * kBarAccEmpty, (acc_it & 1u) ^ 1u, abort, a.status)) break;
        tc_fence_after();
        PW_TRACE_TILE(mode, acc_it, 0);
        const int kc = k_range(tile, ksteps, ksplit).kc;
        bool ok = true;
        for (int s = 0; s < kc; ++s, ++it) {
          const uint32_t stage = it % NST, par = (it / NST) & 1u;
          if (!mbar_wait(bar_base + 8 * (kBarFull + stage), par, abort, a.status)) {
            ok = false;
            break;
          }
          PW_TRACE_STEP(mode, it, 0);
          tc_fence_after();
          const uint32_t a_addr = sbase + kOffA + stage * kAStage;
          const uint32_t b_addr = sbase + kOffB + stage * kBStage;
          issue_kstep(tmem_base, smem_desc(a_addr), smem_desc(a_addr + 32), smem_desc(b_addr),
                      smem_desc(b_addr + 32), smem_desc(b_addr + kBHalf),
                      smem_desc(b_addr + kBHalf + 32), id0, id1, s == 0, n1 > 0,
                      bar_base + 8 * (kBarEmpty + stage));
          issued = true;
          PW_TRACE_STEP(mode, it, 1);
        }
        if (!ok) break;
        mma_commit(bar_base + 8 * kBarAccFull);
        PW_TRACE_TILE(mode, acc_it, 1);
        ++acc_it;
      }
      if (*abort && issued) {
        // wait for every MMA issued so far before TMEM is released
        mma_commit(bar_base + 8 * kBarFinal);
        for (uint32_t i = 0; i < kSpinLimit && !mbar_try(bar_base + 8 * kBarFinal, 0); ++i) {
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------- gather / combine

// xg[pos][c] = fp16(hidden[perm[pos] / k][c] * 2^-e) and scale[pos] = 2^e,
// e putting the row's largest magnitude in [1, 2) (clamped to [-126, 126]);
// positions past the routed pairs are zero with scale 1.  One warp per row
// (two passes over the row: its maximum, then the scaled fp16 values, 8
// columns per lane and step).  Also resets the GEMMs' tile counters.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ hidden,
                                                     const int32_t* __restrict__ perm,
                                                     const int32_t* __restrict__ offsets, int E,
                                                     int k, int H, int n_pairs,
                                                     __half* __restrict__ xg,
                                                     float* __restrict__ xscale,
                                                     int32_t* __restrict__ counters) {
  if (blockIdx.x == 0 && threadIdx.x < 2) counters[threadIdx.x] = 0;
  const int lane = threadIdx.x & 31;
  const int valid = offsets[E];
  const int warps = static_cast<int>(gridDim.x) * (blockDim.x >> 5);
  for (int pos = static_cast<int>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); pos < n_pairs;
       pos += warps) {
    __half* dst = xg + static_cast<long long>(pos) * H;
    if (pos >= valid) {
      for (int c = lane * 8; c < H; c += 256) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
      if (lane == 0) xscale[pos] = 1.f;
      continue;
    }
    const uint16_t* src = hidden + static_cast<long long>(perm[pos] / k) * H;
    uint32_t m = 0;   // bits of |x|: non-negative floats order like their bit patterns
    for (int c = lane * 8; c < H; c += 256) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + c));
      const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m = max(m, max(wv[j] & 0x7FFFu, (wv[j] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    int e = static_cast<int>((m >> 7) & 0xFFu) - 127;   // exponent of the largest bf16 magnitude
    e = min(max(e, -126), 126);
    const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    for (int c = lane * 8; c < H; c += 256) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + c));
      const uint16_t* b = reinterpret_cast<const uint16_t*>(&raw);
      __half2 h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        h[j] = __floats2half2_rn(bf16_bits_to_float(b[2 * j]) * down, bf16_bits_to_float(b[2 * j + 1]) * down);
      *reinterpret_cast<uint4*>(dst + c) = *reinterpret_cast<const uint4*>(h);
    }
    if (lane == 0) xscale[pos] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y_ws,
                                                      const float* __restrict__ y_ws2,
                                                      const int32_t* __restrict__ ids,
                                                      const float* __restrict__ wts, int T, int k,
                                                      int E, int H, float* __restrict__ out) {
  // four consecutive columns per thread (H is a multiple of 32); a row's
  // ids and weights are shared by its threads (L1 hits).  With y_ws2 the
  // down GEMM split K in two: a pair's row is the sum of its two parts.
  const int H4 = H / 4;
  const long long total = static_cast<long long>(T) * H4;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H4);
    const int c4 = static_cast<int>(i - static_cast<long long>(t) * H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int p = t * k + j;
      const int e = __ldg(ids + p);
      if (e < 0 || e >= E) continue;
      const float w = __ldg(wts + p);
      float4 v = __ldcs(reinterpret_cast<const float4*>(y_ws + static_cast<long long>(p) * H) + c4);
      if (y_ws2) {
        const float4 v2 =
            __ldcs(reinterpret_cast<const float4*>(y_ws2 + static_cast<long long>(p) * H) + c4);
        v.x += v2.x;
        v.y += v2.y;
        v.z += v2.z;
        v.w += v2.w;
      }
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    reinterpret_cast<float4*>(out)[i] = acc;
  }
}

// ---------------------------------------------------------------- host side

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  int32_t* counters;   // [2] tile counters of the two GEMM launches
  int32_t* offsets;
  int32_t* perm;
  float* xscale;       // [P] 2^e of each gathered row
  __half* xg;
  __half* h;
  float* y;
  float* y2;   // the down GEMM's second K half
};

WsLayout carve_ws(void* ws, const pw_moe_shape& s) {
  const size_t P = static_cast<size_t>(s.T) * s.k;
  char* p = static_cast<char*>(ws);
  WsLayout w;
  w.counters = reinterpret_cast<int32_t*>(p);
  p += 256;
  w.offsets = reinterpret_cast<int32_t*>(p);
  p += round256(sizeof(int32_t) * (s.E + 1));
  w.perm = reinterpret_cast<int32_t*>(p);
  p += round256(sizeof(int32_t) * P);
  w.xscale = reinterpret_cast<float*>(p);
  p += round256(sizeof(float) * P);
  w.xg = reinterpret_cast<__half*>(p);
  p += round256(2 * P * s.H);
  w.h = reinterpret_cast<__half*>(p);
  p += round256(2 * P * s.I);
  w.y = reinterpret_cast<float*>(p);
  p += round256(4 * P * s.H);
  w.y2 = reinterpret_cast<float*>(p);
  return w;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D fp16 [rows][cols] row-major, box {BK cols, BNH rows}, 64-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int rows, int cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {BK, BNH};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The >48 KB shared-memory opt-in of both GEMM instantiations, set once per
// device.
cudaError_t configure_gemm() {
  cudaError_t e = cudaFuncSetAttribute(dq_gemm_kernel<kGateUp>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dq_gemm_kernel<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmemBytes));
}

}  // namespace

namespace {

// ---------------------------------------------------------------- checks
//
// The dequant warps' index extraction and LUT lookups, run on a whole block
// and written back in column order, for a bit-exact comparison with the
// format's definition.

// One thread per (row n, word column w): both 16-column halves.
template <int Q>
__global__ void __launch_bounds__(256) half_index_check_kernel(const uint32_t* __restrict__ planes,
                                                               int N, int KW, uint8_t* __restrict__ idx,
                                                               const BitConsts bc) {
  const long long total = static_cast<long long>(N) * KW;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long wcol = i / N, n = i % N;
    uint32_t P[Q];
#pragma unroll
    for (int p = 0; p < Q; ++p) P[p] = planes[p * total + wcol * N + n];
    uint8_t* row = idx + n * (32LL * KW) + 32 * wcol;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t ib[4];
      planes_to_index_half<Q>(P, half ? 0x7362u : 0x5140u, ib, bc);
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          row[16 * half + 4 * m + j] = static_cast<uint8_t>((ib[m] >> (8 * j)) & 255u);
    }
  }
}

// One CTA of 128 threads per 128 rows, the dequant warps' LUT layout (entry
// v of a row at v * 256 + slot, four rows per line): each thread loads its
// row's whole LUT, then dequantises every word column of it.
template <int Q>
__global__ void __launch_bounds__(128) half_dequant_check_kernel(const uint32_t* __restrict__ planes,
                                                                 const uint16_t* __restrict__ lut,
                                                                 int N, int KW,
                                                                 float* __restrict__ out,
                                                                 const BitConsts bc) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t slot = static_cast<uint32_t>((w >> 1) * 128 + lane * 4 + (w & 1) * 2);
  const long long plane = static_cast<long long>(N) * KW;
  for (int m0 = blockIdx.x * 128; m0 < N; m0 += gridDim.x * 128) {
    const int row = m0 + 32 * w + lane;
    __syncthreads();   // the previous rows' lookups are done
    if (row < N)
      for (int part = 0; part < 4; ++part) load_lut<Q>(lut, row, slot, part);
    __syncthreads();
    if (row >= N) continue;
    for (int wcol = 0; wcol < KW; ++wcol) {
      uint32_t P[Q];
#pragma unroll
      for (int p = 0; p < Q; ++p) P[p] = planes[p * plane + static_cast<long long>(wcol) * N + row];
      float* dst = out + static_cast<long long>(row) * (32LL * KW) + 32 * wcol;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t ib[4];
        planes_to_index_half<Q>(P, half ? 0x7362u : 0x5140u, ib, bc);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t packed[4];
          dequant_chunk(ib, cc, slot, packed);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 h2 = *reinterpret_cast<const __half2*>(&packed[i]);
            dst[16 * half + 8 * cc + 2 * i] = __low2float(h2);
            dst[16 * half + 8 * cc + 2 * i + 1] = __high2float(h2);
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_half_index_check(const uint32_t* planes, int N, int K, int q, uint8_t* idx,
                                    cudaStream_t s) {
  const BitConsts bc = make_bit_consts();
  const long long total = static_cast<long long>(N) * (K / 32);
  const int grid = static_cast<int>(std::min<long long>((total + 255) / 256, 64LL * sm_count()));
  const int KW = K / 32;
  switch (q) {
    case 3: half_index_check_kernel<3><<<grid, 256, 0, s>>>(planes, N, KW, idx, bc); break;
    case 4: half_index_check_kernel<4><<<grid, 256, 0, s>>>(planes, N, KW, idx, bc); break;
    case 5: half_index_check_kernel<5><<<grid, 256, 0, s>>>(planes, N, KW, idx, bc); break;
    case 6: half_index_check_kernel<6><<<grid, 256, 0, s>>>(planes, N, KW, idx, bc); break;
    case 8: half_index_check_kernel<8><<<grid, 256, 0, s>>>(planes, N, KW, idx, bc); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_half_dequant_check(const uint32_t* planes, const uint16_t* lut, int N, int K,
                                      int q, float* out, cudaStream_t s) {
  const BitConsts bc = make_bit_consts();
  const int KW = K / 32;
  const int grid = std::min((N + 127) / 128, 2 * sm_count());
  cudaError_t e = cudaSuccess;
#define PW_HDQ(QQ)                                                                                \
  do {                                                                                            \
    e = cudaFuncSetAttribute(half_dequant_check_kernel<QQ>,                                       \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kLutBytes)); \
    if (e != cudaSuccess) return e;                                                               \
    half_dequant_check_kernel<QQ><<<grid, 128, kLutBytes, s>>>(planes, lut, N, KW, out, bc);     \
  } while (0)
  switch (q) {
    case 3: PW_HDQ(3); break;
    case 4: PW_HDQ(4); break;
    case 5: PW_HDQ(5); break;
    case 6: PW_HDQ(6); break;
    case 8: PW_HDQ(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef PW_HDQ
  return cudaGetLastError();
}

int prefill_ws_section(const pw_moe_shape& shape, int section, size_t* offset, size_t* bytes) {
  const size_t P = static_cast<size_t>(shape.T) * shape.k;
  // offsets from any 256-aligned base
  char* const base = reinterpret_cast<char*>(static_cast<uintptr_t>(1) << 20);
  const WsLayout w = carve_ws(base, shape);
  switch (section) {
    case 0: *offset = reinterpret_cast<const char*>(w.offsets) - base; *bytes = 4 * (static_cast<size_t>(shape.E) + 1); return 0;
    case 1: *offset = reinterpret_cast<const char*>(w.perm) - base; *bytes = 4 * P; return 0;
    case 2: *offset = reinterpret_cast<const char*>(w.xg) - base; *bytes = 2 * P * shape.H; return 0;
    case 3: *offset = reinterpret_cast<const char*>(w.xscale) - base; *bytes = 4 * P; return 0;
    default: return -1;
  }
}

// The trace of the last traced launch (zeros if the library was built without
// PW_TRACE); returns false when tracing is compiled out.
bool gemm_trace_read(void* host, size_t bytes, cudaError_t* err) {
#ifdef PW_TRACE
  *err = cudaMemcpyFromSymbol(host, g_trace, sizeof(GemmTrace) < bytes ? sizeof(GemmTrace) : bytes);
  return true;
#else
  (void)host;
  (void)bytes;
  *err = cudaSuccess;
  return false;
#endif
}

size_t gemm_trace_bytes() { return sizeof(GemmTrace); }

// Clears the trace record before a traced launch (nothing without PW_TRACE).
cudaError_t gemm_trace_clear(cudaStream_t stream) {
#ifdef PW_TRACE
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_trace);
  if (e != cudaSuccess) return e;
  return cudaMemsetAsync(p, 0, sizeof(GemmTrace), stream);
#else
  (void)stream;
  return cudaSuccess;
#endif
}

cudaError_t launch_wait_check_mbar(int32_t* status, uint32_t polls, cudaStream_t s) {
  mbar_wait_check_kernel<<<1, 32, 0, s>>>(status, polls);
  return cudaGetLastError();
}

size_t heavy_scratch_bytes(const pw_moe_shape& s) {
  const size_t P = static_cast<size_t>(s.T) * s.k;
  return 256 + round256(sizeof(float) * P) + round256(2 * P * s.H) + round256(2 * P * s.I);
}

// Decode calls with experts that hold many pairs: those experts run through
// the gather and the two GEMM kernels here, on the decode path's grouping,
// and write their pairs' rows of y; the decode kernels take the rest and
// combine.
cudaError_t launch_heavy(const LayerArgs& la, const int32_t* offsets, const int32_t* perm, float* y,
                         void* scratch, int min_tokens, cudaStream_t stream) {
  cudaError_t e0 = setup_once(kSetupGemm, configure_gemm);
  if (e0 != cudaSuccess) return e0;
  const int sms = sm_count();
  const int n_pairs = la.T * la.k;
  const size_t P = static_cast<size_t>(n_pairs);
  char* p = static_cast<char*>(scratch);
  int32_t* counters = reinterpret_cast<int32_t*>(p);
  p += 256;
  float* xscale = reinterpret_cast<float*>(p);
  p += round256(sizeof(float) * P);
  __half* xg = reinterpret_cast<__half*>(p);
  p += round256(2 * P * la.H);
  __half* h = reinterpret_cast<__half*>(p);
  const int gblocks = static_cast<int>(std::min<long long>((n_pairs + 7) / 8, 32LL * sms));
  gather_kernel<<<gblocks, 256, 0, stream>>>(la.hidden, perm, offsets, la.E, la.k, la.H, n_pairs, xg,
                                             xscale, counters);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap map_x, map_h;
  if (!make_map(&map_x, xg, n_pairs, la.H) || !make_map(&map_h, h, n_pairs, la.I))
    return cudaErrorInvalidValue;
  GemmArgs g;
  g.H = la.H;
  g.I = la.I;
  g.E = la.E;
  g.k = la.k;
  g.n_pairs = n_pairs;
  g.table = la.table;
  g.offsets = offsets;
  g.perm = perm;
  g.xscale = xscale;
  g.h_ws = h;
  g.y_ws = y;
  g.y_ws2 = nullptr;
  g.ksplit = 1;   // the decode path's combine reads one y
  g.status = la.status;
  g.min_tokens = min_tokens;
  const int grid = sms;
  const BitConsts bc = make_bit_consts();
  g.tile_counter = counters;
  if ((e = gemm_trace_clear(stream)) != cudaSuccess) return e;
  dq_gemm_kernel<kGateUp><<<grid, kThreads, kSmemBytes, stream>>>(g, map_x, bc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  g.tile_counter = counters + 1;
  dq_gemm_kernel<kDown><<<grid, kThreads, kSmemBytes, stream>>>(g, map_h, bc);
  return cudaGetLastError();
}

size_t prefill_workspace_bytes(const pw_moe_shape& s) {
  const size_t P = static_cast<size_t>(s.T) * s.k;
  return 256 + round256(sizeof(int32_t) * (s.E + 1)) + round256(sizeof(int32_t) * P) +
         round256(sizeof(float) * P) + round256(2 * P * s.H) + round256(2 * P * s.I) +
         2 * round256(4 * P * s.H);
}

bool prefill_shape_ok(const pw_moe_shape& s) {
  return s.H % BM == 0 && s.I % 64 == 0 && s.E <= kMaxExperts;
}

int prefill_min_pairs(const pw_moe_shape& s) { return prefill_shape_ok(s) ? 1024 : INT_MAX; }

cudaError_t launch_prefill(const LayerArgs& la, void* ws, cudaStream_t stream) {
  cudaError_t e0 = setup_once(kSetupGemm, configure_gemm);
  if (e0 != cudaSuccess) return e0;
  const int sms = sm_count();
  pw_moe_shape s{la.T, la.H, la.I, la.E, la.k};
  const int n_pairs = la.T * la.k;
  if (n_pairs == 0) return cudaSuccess;
  WsLayout w = carve_ws(ws, s);
  cudaError_t e = launch_permute(la.topk_ids, n_pairs, la.E, w.offsets, w.perm, nullptr, la.status,
                                 stream, la.logits, la.k, la.route_wts);
  if (e != cudaSuccess) return e;
  if ((e = launch_routing_stats(la, stream)) != cudaSuccess) return e;
  const int gblocks = static_cast<int>(std::min<long long>((n_pairs + 7) / 8, 32LL * sms));
  gather_kernel<<<gblocks, 256, 0, stream>>>(la.hidden, w.perm, w.offsets, la.E, la.k, la.H,
                                             n_pairs, w.xg, w.xscale, w.counters);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  CUtensorMap map_x, map_h;
  if (!make_map(&map_x, w.xg, n_pairs, la.H) || !make_map(&map_h, w.h, n_pairs, la.I))
    return cudaErrorInvalidValue;
  GemmArgs g;
  g.H = la.H;
  g.I = la.I;
  g.E = la.E;
  g.k = la.k;
  g.n_pairs = n_pairs;
  g.table = la.table;
  g.offsets = w.offsets;
  g.perm = w.perm;
  g.xscale = w.xscale;
  g.h_ws = w.h;
  g.y_ws = w.y;
  g.y_ws2 = w.y2;
  g.ksplit = 1;
  g.status = la.status;
  g.min_tokens = 1;
  const int grid = sms;
  const BitConsts bc = make_bit_consts();
  g.tile_counter = w.counters;
  if ((e = gemm_trace_clear(stream)) != cudaSuccess) return e;
  if ((e = record_timing(g_timing.before, stream)) != cudaSuccess) return e;
  dq_gemm_kernel<kGateUp><<<grid, kThreads, kSmemBytes, stream>>>(g, map_x, bc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = record_timing(g_timing.after, stream)) != cudaSuccess) return e;
  // The down GEMM has H/128 row tiles per expert, too few to fill the SMs
  // evenly (a Mixtral-shaped call: 512 tiles on 152 SMs, 3.4 rounds); its K
  // (= I) is long, so each weight tile's K range is split over two tiles
  // whose partial sums land in y and y2 and meet in the combine.
  g.tile_counter = w.counters + 1;
  g.ksplit = (la.I / BK >= 2) ? 2 : 1;
  dq_gemm_kernel<kDown><<<grid, kThreads, kSmemBytes, stream>>>(g, map_h, bc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long cwork = static_cast<long long>(la.T) * (la.H / 4);
  const int cblocks = static_cast<int>(std::min<long long>((cwork + 255) / 256, 32LL * sms));
  combine_kernel<<<cblocks, 256, 0, stream>>>(w.y, g.ksplit == 2 ? w.y2 : nullptr, la.topk_ids,
                                              la.topk_weights, la.T, la.k, la.E, la.H, la.out);
  return cudaGetLastError();
}

}  // namespace pw
