// Fused mixed-precision MoE layer, decode path (few tokens per expert).
//
// PagedWeight, "Core components" 3 (fused mixed-precision kernel): every
// linear block's bitplanes and LUT are read directly, each block at its own
// committed bitwidth q_i, inside one fused operation.  Three launches, chained
// with programmatic dependent launch so that each one's start-up overlaps the
// previous one's tail:
//
//   prep:    CTA 0 groups the (token, expert) pairs by expert (stable), lists
//            the routed experts largest-bitwidth first (so the costliest
//            tiles are scheduled first) with each one's page-table entry,
//            and resets the tile counters; the other CTAs widen the hidden
//            states to fp32 and zero `out`.  In small calls it is launched
//            early too, behind the previous call's down kernel.
//   [heavy]  in calls of at least kHybridMinTokens tokens, experts holding
//            at least kHeavyMinTokens pairs are left out of
//            those lists: the tcgen05 GEMM kernels of the prefill path run
//            them (gather, gate_up, down -> y) between prep and gate_up, so
//            their planes are read and dequantised once instead of once per
//            group of 4 tokens.
//   gate_up: persistent CTAs take tiles (routed expert, 32 gate/up row pairs)
//            from an atomic counter: read the top q planes of gate rows i and
//            up rows I+i, rebuild the q-bit codes, look them up in each row's
//            LUT, dot with the expert's tokens (fp32), h = SiLU(g) * u.
//   down:    persistent CTAs take tiles (routed expert, 64 down rows): same
//            read of the down block, dot with h -> y for each pair.  When
//            the down tiles are short (K = I <= kEarlyDownMaxI) a down tile
//            waits only for its own expert's gate_up tiles (a per-expert
//            counter that each finished gate_up tile increments after a
//            fence), so down tiles fill the SMs that the gate_up tail leaves
//            idle; long down tiles would slow the last gate_up tiles they
//            share an SM with, so they wait for the whole gate_up grid.  The
//            last tile to finish a 64-row range (arrival counter) forms
//            out[t] = sum_j w_tj * y[t*k + j] over the range in j order, so
//            the output is deterministic.  A long down K (I >= 8192) in a
//            call whose down tiles fill less than two rounds is split in two
//            halves (decode_down_kernel<2>): two tiles per range, the second
//            half's partial sums in y2, which the combine adds first.
//
// Work inside a CTA: each lane owns one or two rows of the tile; the 8 warps
// split the K columns and their partial sums meet in shared memory.  A warp
// streams its word columns through a 3-stage cp.async ring: per column, one
// word of each of the top q planes per row (a word column of consecutive
// rows is contiguous, so each copy is part of a 128-byte line) plus the 32
// matching activations of up to 4 tokens.  A lane turns its q plane words
// into indices with a register-index / bit-position transpose (swap stages
// of shifts and bit selects, no byte shuffles); the indices come out in a
// fixed permuted column order, and the activations are stored in that same
// order, so every product still pairs a weight with its own column.  Two
// lookup forms, by bitwidth:
//   q = 3, 4  nibble indices; one byte of them is a pair of columns, looked
//             up in a pair table of the row (2^2q entries, each the fp16
//             pair {LUT[a], LUT[b]}) with one byte permute and one shared
//             load per two weights; products are packed fp16 pairs against
//             fp16 activations, summed in fp16 over the 8 pairs of each
//             16-column half of a word column and then added to fp32
//             accumulators with that half's power-of-two scale (activations
//             are stored per 16 columns as x * 2^-e with max |x * 2^-e| in
//             [1, 2), so no fp16 value overflows and the fp16 partial sums
//             keep their relative precision);
//   q = 5, 6, 8  byte indices, one lookup per weight in the row's fp32 LUT;
//             products accumulate as packed fp32 pairs against fp32
//             activations.
// Every lookup of lane L hits bank L (the tables are lane-interleaved).
// q = 4 and q = 8 blocks stream one row per lane so that their tables fit.
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "pw_bits.cuh"
#include "pw_internal.cuh"
#include "pw_router.cuh"

namespace pw {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPairsPerTile = 32;   // gate_up tile: 32 gate rows + their 32 up rows
constexpr int kDownRows = 64;       // down tile: two 32-row groups
constexpr int kTG = 4;              // tokens per pass over the weights
// the reduction of a token group uses warps 0..kTG-1, so the last warp is
// free to claim the next gate_up tile meanwhile
static_assert(kTG < kWarps, "the claiming warp must not reduce");
constexpr int kStages = 3;          // per-warp cp.async ring depth (word columns)
constexpr int kMaxPairs = 4096;     // T*k limit of this path
constexpr int kMaxExperts = 1024;
constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;

// One ring stage holds one word column (32 weights) of every streamed row:
// q*R plane words per lane (at most 12: q <= 6 with two row slots, or q = 8
// with one) and the matching 32 activations of up to kTG tokens.
constexpr int kStagePlaneBytes = 12 * 128;
constexpr int kStageBytes = kStagePlaneBytes + kTG * 128;

// Shared memory (bytes).  LUT region first.  Two layouts:
//   paired  (two row slots): entry v of slot g for lane L at v*256 + g*128
//           + L*4, so one byte permute of the index byte forms the offset;
//   compact (one row slot):  entry v for lane L at v*128 + L*4 (the permute
//           gives v*256 + L*8, halved by one shift).
// Either way a lane's lookups always hit bank L.  An entry is an fp32 weight
// (q = 5, 6, 8) or an fp16 pair of weights indexed by two nibble indices
// (q = 3 paired, q = 4 compact).
constexpr int kLutBytes = 32768;
constexpr int kRingBytes = kWarps * kStages * kStageBytes;
constexpr int kRedBytes = kWarps * kTG * 2 * 32 * 4;
constexpr int kOffRing = kLutBytes;
constexpr int kOffRed = kOffRing + kRingBytes;
constexpr int kOffMisc = kOffRed + kRedBytes;
constexpr size_t kSmemBytes = kOffMisc + 64;

// The dynamic shared memory of the decode kernels.  Hot-loop accesses index
// this symbol directly with 32-bit offsets, so they compile to shared loads
// with register + immediate addressing.
extern __shared__ __align__(16) unsigned char g_dsmem[];

// ---------------------------------------------------------------- trace
// With PW_TRACE (the traced build) the gate_up kernel records, for every
// kDTraceStride-th CTA (up to kDTraceCtas of them) and its first kDTraceTiles
// tiles: the tile's start and end (%globaltimer ns); the SM cycles (clock64)
// that thread 0 spent on the slot descriptor (with the previous tile's
// release), on the passes' set-up (LUT fetch, ring prime, table build, up to
// the barrier after it), on the token groups' column loops (up to the barrier
// after the partial sums) and on their reduction and h stores; the tile's q
// and pair count; the set-up's parts (issuing the LUT loads and the first
// ring copies; waiting for its LUT words and building its share of the
// tables; the barrier after the build); and per traced CTA its SM and exit
// time.  Thread 0 alone writes; misc[15] holds the current tile's record
// index (-1: not traced).  The launch path clears the record before each
// gate_up launch.  Without PW_TRACE every hook is empty.
constexpr int kDTraceTiles = 32, kDTraceCtas = 16, kDTraceFields = 10;
struct DecodeTrace {
  // start ns, end ns, descriptor, set-up, columns, reduction + store (cycles),
  // q + 256 * pairs, set-up parts: issue, LUT wait + build, barrier (cycles)
  unsigned long long tile[kDTraceCtas][kDTraceTiles][kDTraceFields];
  unsigned long long cta[kDTraceCtas][2];   // SM id + 1 (0: not traced), exit ns
};
#ifdef PW_TRACE
constexpr int kDTraceStride = 19;
__device__ DecodeTrace g_dtrace;
__device__ __forceinline__ unsigned long long dtrace_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int dtrace_cta() {
  const int b = static_cast<int>(blockIdx.x);
  return (b % kDTraceStride == 0 && b / kDTraceStride < kDTraceCtas) ? b / kDTraceStride : -1;
}
__device__ __forceinline__ unsigned long long* dtrace_field(int rec, int k) {
  return &g_dtrace.tile[0][0][0] + static_cast<long long>(rec) * kDTraceFields + k;
}
#define PW_DTRACE_TILE_BEGIN(s, j, clk)                                                \
  long long clk = 0;                                                                    \
  if (threadIdx.x == 0) {                                                               \
    const int c_ = dtrace_cta();                                                        \
    (s).misc[15] = (c_ >= 0 && (j) < kDTraceTiles) ? c_ * kDTraceTiles + (j) : -1;      \
    if ((s).misc[15] >= 0) {                                                            \
      *dtrace_field((s).misc[15], 0) = dtrace_ns();                                     \
      clk = clock64();                                                                  \
    }                                                                                   \
  }
#define PW_DTRACE_MARK(clk) const long long clk = threadIdx.x == 0 ? clock64() : 0
// a reduction (no value returned), so that thread 0 does not wait for the
// record's old value
#define PW_DTRACE_ADD(s, k, clk)                                                       \
  do {                                                                                  \
    if (threadIdx.x == 0 && (s).misc[15] >= 0)                                          \
      atomicAdd(dtrace_field((s).misc[15], (k)),                                        \
                static_cast<unsigned long long>(clock64() - (clk)));                    \
  } while (0)
#define PW_DTRACE_TILE_END(s, q, pairs)                                                \
  do {                                                                                  \
    if (threadIdx.x == 0 && (s).misc[15] >= 0) {                                        \
      *dtrace_field((s).misc[15], 1) = dtrace_ns();                                     \
      *dtrace_field((s).misc[15], 6) = (q) + 256ull * (pairs);                          \
    }                                                                                   \
  } while (0)
#define PW_DTRACE_EXIT()                                                               \
  do {                                                                                  \
    const int c_ = dtrace_cta();                                                        \
    if (threadIdx.x == 0 && c_ >= 0) {                                                  \
      unsigned sm_;                                                                     \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                                  \
      g_dtrace.cta[c_][0] = sm_ + 1ull;                                                 \
      g_dtrace.cta[c_][1] = dtrace_ns();                                                \
    }                                                                                   \
  } while (0)
#else
#define PW_DTRACE_TILE_BEGIN(s, j, clk) do { } while (0)
#define PW_DTRACE_MARK(clk) do { } while (0)
#define PW_DTRACE_ADD(s, k, clk) do { } while (0)
#define PW_DTRACE_TILE_END(s, q, pairs) do { } while (0)
#define PW_DTRACE_EXIT() do { } while (0)
#endif

struct SmemPtrs {
  unsigned char* lut;
  unsigned char* ring;
  float* red;
  int* misc;
};

__device__ __forceinline__ SmemPtrs carve(unsigned char* base) {
  SmemPtrs s;
  s.lut = base;
  s.ring = base + kOffRing;
  s.red = reinterpret_cast<float*>(base + kOffRed);
  s.misc = reinterpret_cast<int*>(base + kOffMisc);
  return s;
}

// One routed expert's share of a kernel, written by the prep launch so that a
// tile needs one dependent load: the expert, its grouped pair positions and
// the page-table entry of the kernel's block (copied at prep time; the table
// changes only between calls).
struct SlotInfo {
  int32_t e;        // expert id
  int32_t off;      // first grouped pair position of e
  int32_t ne;       // pairs routed to e
  int32_t q;        // committed bitwidth of the block
  int32_t err;      // 0 if the tiles can run, else the status to latch
  int32_t q_other;  // bitwidth of the expert's other block (gate_up: the down
                    // block, whose form decides how h is stored)
  const uint32_t* planes;
  const uint16_t* lut;
  int32_t rows[4];  // hidden-state rows of the expert's first kTG pairs (the
                    // last one repeated), so a pass's first copies need no
                    // dependent load of perm
};

static_assert(sizeof(SlotInfo) == 56, "slot descriptor layout");

// Workspace of one decode call.
// Activations come in two forms, matching the two lookup forms (the column
// order inside each group of 32 is the one the index form produces):
//   fp32 form  float [rows][K], column c of a group at byte_form_position(c);
//   fp16 form  one 80-byte record per (row, group of 32 columns): 32 fp16
//              values x * 2^-e at nibble_form_position(c), where e is that of
//              the column's half of the group (columns 0-15 or 16-31: e puts
//              the half's largest |x * 2^-e| in [1, 2)); then the floats 2^e
//              of the two halves at bytes 64 and 68, then padding.
constexpr int kRecBytes = 80;

struct DecodeWs {
  float* xs;       // [T][H]   hidden states, fp32 form
  char* xp;        // [T][H/32] records: hidden states, fp16 form
  float* hs;       // [P][I]   SiLU(g) * u by grouped pair position, fp32 form
  char* hp;        // [P][I/32] records: the same in fp16 form (down blocks at q <= 4)
  float* y;        // [P][H]   expert output, by pair id (with dn_ks = 2: its first K half)
  float* y2;       // [P][H]   the second K half's partial sums (dn_ks = 2), else unused
  int* offsets;    // [E+1]    expert e owns grouped positions offsets[e] .. offsets[e+1]
  int* perm;       // [P]      grouped position -> pair id
  SlotInfo* routed_gu;  // [E] routed experts, gate_up bitwidth descending
  SlotInfo* routed_dn;  // [E] routed experts, down bitwidth descending
  int* ctl;        // [0] routed expert count, [1] gate_up tile counter, [2] down tile counter
  int* arrive;     // [H/32]   per 64-row range: down tiles finished
  int* gu_done;    // [P]      gate_up tiles finished per token group, indexed by the
                   //          group's first grouped position (released by a fence)
  int heavy_min;   // experts with at least this many pairs are left to the GEMM kernels (0: none)
  int early_next;  // 1: the down grid leaves SM slots free, so it lets the next launch start early
  int dn_ks;       // K parts per down row range: 1, or 2 (long K in calls with few down tiles)
};

// Rows streamed by one pass: lane L of row slot g owns row
// seg[g][L >> 4] + (L & 15), i.e. each slot is two 16-row segments.
template <int R>
struct PassRows {
  int seg[R][2];
};

// One expert's share of a call.
struct ExpertWork {
  int e;    // expert id
  int off;  // first grouped pair position of e
  int ne;   // pairs routed to e
};

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int R>
__device__ __forceinline__ int seg_base(const PassRows<R>& pr, int g, int seg) {
  const int a = seg ? pr.seg[0][1] : pr.seg[0][0];
  if (R == 1) return a;
  const int b = seg ? pr.seg[R - 1][1] : pr.seg[R - 1][0];
  return g ? b : a;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Lookup form of a block at bitwidth Q: pair tables with nibble indices for
// Q <= 4 (fp16 products), fp32 tables with byte indices otherwise.
template <int Q>
struct Form {
  static constexpr bool kPair = Q <= 4;
  // bytes of one token's activations in a ring stage (a record, or 32 floats)
  static constexpr int kXBytes = kPair ? kRecBytes : 128;
  static constexpr int kXChunks = kXBytes / 16;
};

// Power-of-two group scale: e with m * 2^-e in [1, 2) for the group's largest
// magnitude m (clamped so that 2^e and 2^-e are normal floats).
__device__ __forceinline__ int group_exponent(float m) {
  const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  return min(max(e, -126), 126);
}

__device__ __forceinline__ float exp2i(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// fp32 tables (Q = 5, 6, 8): the LUT rows of one pass into shared memory
// (layouts above), in two steps so that the round trip overlaps other set-up
// work: lut_fetch issues every global load of the thread (up to four 16-byte
// pieces of 8 fp16 entries) into registers, lut_store converts and stores
// them.  A warp's stores hit 32 banks.
template <int Q, int R>
struct LutPieces {
  static constexpr int kEnt = 1 << Q;
  static constexpr int kVecPerRow = kEnt / 8;
  static constexpr int kPerSlot = 32 * kVecPerRow;
  static constexpr int kTotal = R * kPerSlot;
  static constexpr int kPer = (kTotal + kThreads - 1) / kThreads;
  uint4 raw[kPer];
};

template <int Q, int R>
__device__ __forceinline__ void lut_fetch(const uint16_t* lut, const PassRows<R>& pr,
                                          LutPieces<Q, R>& lp) {
  using L = LutPieces<Q, R>;
#pragma unroll
  for (int j = 0; j < L::kPer; ++j) {
    const int i = threadIdx.x + j * kThreads;
    if (i < L::kTotal) {
      const int g = i / L::kPerSlot, rem = i % L::kPerSlot;
      const int lane = rem & 31, vec = rem >> 5;
      const int row = seg_base<R>(pr, g, lane >> 4) + (lane & 15);
      lp.raw[j] = __ldg(reinterpret_cast<const uint4*>(lut + static_cast<long long>(row) * L::kEnt +
                                                       vec * 8));
    }
  }
}

template <int Q, int R, bool COMPACT>
__device__ __forceinline__ void lut_store(const LutPieces<Q, R>& lp) {
  using L = LutPieces<Q, R>;
#pragma unroll
  for (int j = 0; j < L::kPer; ++j) {
    const int i = threadIdx.x + j * kThreads;
    if (i < L::kTotal) {
      const int g = i / L::kPerSlot, rem = i % L::kPerSlot;
      const int lane = rem & 31, vec = rem >> 5;
      const __half* h = reinterpret_cast<const __half*>(&lp.raw[j]);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int v = vec * 8 + jj;
        const int off = COMPACT ? v * 128 + lane * 4 : v * 256 + g * 128 + lane * 4;
        *reinterpret_cast<float*>(g_dsmem + off) = __half2float(h[jj]);
      }
    }
  }
}

// Pair tables (Q = 3, 4): entry v = a + 16 b of a row holds the fp16 pair
// {LUT[a], LUT[b]} (low half a), looked up by one byte of nibble indices.
// kTPR threads build each row's table: lane L of warp W takes row L of slot
// W % R and the share c = W / R of its entries (those whose high nibble b is
// in that share), so that a warp's stores hit 32 different rows and banks,
// and its fetches read 32 consecutive rows' LUTs (2^Q fp16 values each, one
// or two 16-byte loads).  Only pairs of valid indices are written (Q = 3:
// a, b < 8).
template <int Q, int R>
struct PairLutPieces {
  static constexpr int kTPR = 8 / R;                 // threads per row (R*32 rows)
  static constexpr int kBPT = (1 << Q) / kTPR;       // b values per thread
  static constexpr int kWords = (1 << Q) / 2;        // u32 words of a row's LUT
  uint32_t w[kWords];
};

template <int Q, int R>
__device__ __forceinline__ void pair_lut_fetch(const uint16_t* lut, const PassRows<R>& pr,
                                               PairLutPieces<Q, R>& lp) {
  using L = PairLutPieces<Q, R>;
  if (threadIdx.x >= 256) return;   // 256 threads build the tables
  const int g = (threadIdx.x >> 5) % R, lane = threadIdx.x & 31;
  const int row = seg_base<R>(pr, g, lane >> 4) + (lane & 15);
  const uint4* src = reinterpret_cast<const uint4*>(lut + static_cast<long long>(row) * (1 << Q));
#pragma unroll
  for (int v = 0; v < L::kWords / 4; ++v) {
    const uint4 q4 = __ldg(src + v);
    lp.w[4 * v] = q4.x;
    lp.w[4 * v + 1] = q4.y;
    lp.w[4 * v + 2] = q4.z;
    lp.w[4 * v + 3] = q4.w;
  }
}

// Largest LUT magnitude a pair-table block supports: 16 products of such a
// value with activations below 2 in magnitude stay inside fp16's range.
constexpr uint32_t kPairLutLimitBits = 0x6800u;   // fp16 2048

template <int Q, int R, bool COMPACT>
__device__ __forceinline__ void pair_lut_store(const PairLutPieces<Q, R>& lp, int32_t* status) {
  using L = PairLutPieces<Q, R>;
  if (threadIdx.x >= 256) return;   // 256 threads build the tables
  const int g = (threadIdx.x >> 5) % R, c = (threadIdx.x >> 5) / R, lane = threadIdx.x & 31;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < L::kWords; ++i)
    bad |= ((lp.w[i] & 0x7FFFu) >= kPairLutLimitBits) || (((lp.w[i] >> 16) & 0x7FFFu) >= kPairLutLimitBits);
  if (bad) latch_status(status, PW_ERR_RANGE);
  const uint32_t base = COMPACT ? static_cast<uint32_t>(lane * 4)
                                : static_cast<uint32_t>(g * 128 + lane * 4);
  constexpr uint32_t kStride = COMPACT ? 128u : 256u;
#pragma unroll
  for (int bi = 0; bi < L::kBPT; ++bi) {
    const int b = c * L::kBPT + bi;
    // the word holding LUT[b] (runtime index into the register array)
    uint32_t y = lp.w[0];
#pragma unroll
    for (int i = 1; i < L::kWords; ++i)
      if ((b >> 1) == i) y = lp.w[i];
    const uint32_t hi_sel = (b & 1) ? 0x7600u : 0x5400u;   // high half = LUT[b]
#pragma unroll
    for (int a = 0; a < (1 << Q); ++a) {
      const uint32_t sel = hi_sel | ((a & 1) ? 0x32u : 0x10u);   // low half = LUT[a]
      const uint32_t v = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 4);
      *reinterpret_cast<uint32_t*>(g_dsmem + v * kStride + base) = __byte_perm(lp.w[a >> 1], y, sel);
    }
  }
}

// The LUT of one pass, in the form of bitwidth Q: issued first (fetch), then
// stored once the first ring columns are on their way (store).
template <int Q, int R>
struct PassLut {
  using Pieces = typename std::conditional<Form<Q>::kPair, PairLutPieces<Q, R>, LutPieces<Q, R>>::type;
  Pieces p;
};

template <int Q, int R>
__device__ __forceinline__ void pass_lut_fetch(const uint16_t* lut, const PassRows<R>& pr,
                                               PassLut<Q, R>& pl) {
  if constexpr (Form<Q>::kPair) pair_lut_fetch<Q, R>(lut, pr, pl.p);
  else lut_fetch<Q, R>(lut, pr, pl.p);
}

template <int Q, int R, bool COMPACT>
__device__ __forceinline__ void pass_lut_store(const PassLut<Q, R>& pl, int32_t* status) {
  if constexpr (Form<Q>::kPair) pair_lut_store<Q, R, COMPACT>(pl.p, status);
  else lut_store<Q, R, COMPACT>(pl.p);
}

// The copies one lane issues for every word column: chunk c (16 bytes) of
// a stage is plane p = (c/8)/R, row slot g = (c/8)%R, 16-row segment
// (c/4)%2 and quarter c%4; it lands at stage byte c*16.  Its source is
// planes + src_off + kw*N; the word offsets are fixed for a pass, so they are
// computed once.  Activation chunk lane (< NT * kXChunks): token
// lane / kXChunks, 16-byte piece lane % kXChunks of the token's activations
// for the word column (32 floats, or one fp16 record).
template <int Q, int R, int NT>
struct CopyPlan {
  static constexpr int kChunks = (Q * R * 8 + 31) / 32;
  uint32_t src_off[kChunks];
  const char* x_src;    // token row + piece offset (word column 0)
  uint32_t x_bytes;     // 16, or 0 to zero-fill an absent token
};

template <int Q, int R, int NT>
__device__ __forceinline__ CopyPlan<Q, R, NT> make_copy_plan(long long plane_stride,
                                                             const PassRows<R>& pr,
                                                             const char* const (&xs)[NT],
                                                             int nt, int lane) {
  constexpr int XC = Form<Q>::kXChunks;
  CopyPlan<Q, R, NT> cp;
#pragma unroll
  for (int i = 0; i < CopyPlan<Q, R, NT>::kChunks; ++i) {
    const int c = i * 32 + lane;
    const int pg = c >> 3, seg = (c >> 2) & 1, part = c & 3;
    const int p = pg / R, g = pg % R;
    cp.src_off[i] = (c < Q * R * 8)
                        ? static_cast<uint32_t>(p * plane_stride + seg_base<R>(pr, g, seg) + part * 4)
                        : 0u;
  }
  const int tk = lane / XC, part = lane % XC;
  const bool live = lane < NT * XC && tk < nt;
  const char* base = xs[0];
#pragma unroll
  for (int i = 1; i < NT; ++i)
    if (live && tk == i) base = xs[i];
  cp.x_src = base + part * 16;
  cp.x_bytes = live ? 16u : 0u;
  return cp;
}

// Start the asynchronous copies of word column kw of every streamed row and
// of the matching activations of each token into one ring stage.
template <int Q, int R, int NT>
__device__ __forceinline__ void issue_column(uint32_t stage, const uint32_t* planes, long long N,
                                             const CopyPlan<Q, R, NT>& cp, int kw, int lane) {
  constexpr int XC = Form<Q>::kXChunks;
  const uint32_t col = static_cast<uint32_t>(kw * N);
#pragma unroll
  for (int i = 0; i < CopyPlan<Q, R, NT>::kChunks; ++i) {
    const int c = i * 32 + lane;
    if (c < Q * R * 8) cp_async16(stage + c * 16, planes + (cp.src_off[i] + col), 16);
  }
  if (lane < NT * XC)
    cp_async16(stage + kStagePlaneBytes + lane * 16,
               cp.x_src + (cp.x_bytes ? static_cast<long long>(kw) * Form<Q>::kXBytes : 0),
               cp.x_bytes);
}

__device__ __forceinline__ uint4 lds128(uint32_t off) {
  return *reinterpret_cast<const uint4*>(g_dsmem + off);
}

// Lane L's base offset in the LUT region for row slot g, and the offset of
// the table entry that byte j of an index word selects (one byte permute; in
// the compact layout entries are 128 bytes apart, so the permute's v * 256 +
// 8L is halved).  Shared by the column loops and the lookup check.
template <bool COMPACT>
__device__ __forceinline__ uint32_t lane_base(int g, int lane) {
  return COMPACT ? (static_cast<uint32_t>(lane) << 3)
                 : ((static_cast<uint32_t>(g) << 7) | (static_cast<uint32_t>(lane) << 2));
}

template <bool COMPACT>
__device__ __forceinline__ uint32_t lut_offset(uint32_t word, uint32_t lb, int j) {
  const uint32_t off = __byte_perm(word, lb, 0x6504 | (j << 4));
  return COMPACT ? off >> 1 : off;
}

// One word column from a ring stage, fp32 tables (Q = 5, 6, 8): byte indices
// of each row, one lookup per weight, packed fp32 products.  B[r] byte b is
// column 8b + r, whose activation sits at position 4r + b: the float4 at 4r.
template <int Q, int R, int NT, bool COMPACT>
__device__ __forceinline__ void compute_column_bytes(uint32_t stage, int lane, const BitConsts& bc,
                                                     float2 (&acc)[R][NT]) {
  uint32_t ib[R][8];
#pragma unroll
  for (int g = 0; g < R; ++g) {
    uint32_t cur[Q];
#pragma unroll
    for (int p = 0; p < Q; ++p)
      cur[p] = *reinterpret_cast<const uint32_t*>(g_dsmem + stage + (p * R + g) * 128 + lane * 4);
    planes_to_bytes<Q>(cur, ib[g], bc);
  }
  const uint32_t xa = stage + kStagePlaneBytes;
  uint32_t lb[R];
#pragma unroll
  for (int g = 0; g < R; ++g) lb[g] = lane_base<COMPACT>(g, lane);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float4 xv[NT];
#pragma unroll
    for (int tk = 0; tk < NT; ++tk) {
      const uint4 u = lds128(xa + tk * 128 + r * 16);
      xv[tk] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                           __uint_as_float(u.w));
    }
#pragma unroll
    for (int g = 0; g < R; ++g) {
      float w[4];
#pragma unroll
      for (int b = 0; b < 4; ++b)
        w[b] = *reinterpret_cast<const float*>(g_dsmem + lut_offset<COMPACT>(ib[g][r], lb[g], b));
#pragma unroll
      for (int tk = 0; tk < NT; ++tk) {
        acc[g][tk] = __ffma2_rn(make_float2(w[0], w[1]), make_float2(xv[tk].x, xv[tk].y), acc[g][tk]);
        acc[g][tk] = __ffma2_rn(make_float2(w[2], w[3]), make_float2(xv[tk].z, xv[tk].w), acc[g][tk]);
      }
    }
  }
}

// One word column from a ring stage, pair tables (Q = 3, 4): nibble indices
// of each row; byte j of N[r] pairs columns 8j + r and 8j + 4 + r, whose
// fp16 activations sit at positions 8r + 2j and 8r + 2j + 1: half2 j of the
// 16 bytes at 16r of the token's record.  The fp16 products of each half of
// the word column (8 pairs) are summed in a half2, which is then added to the
// fp32 accumulator with that half's scale 2^e.
template <int Q, int R, int NT, bool COMPACT>
__device__ __forceinline__ void compute_column_pairs(uint32_t stage, int lane, const BitConsts& bc,
                                                     float2 (&acc)[R][NT]) {
  uint32_t nb[R][4];
#pragma unroll
  for (int g = 0; g < R; ++g) {
    uint32_t cur[Q];
#pragma unroll
    for (int p = 0; p < Q; ++p)
      cur[p] = *reinterpret_cast<const uint32_t*>(g_dsmem + stage + (p * R + g) * 128 + lane * 4);
    planes_to_nibbles<Q>(cur, nb[g], bc);
  }
  const uint32_t xa = stage + kStagePlaneBytes;
  uint32_t lb[R];
#pragma unroll
  for (int g = 0; g < R; ++g) lb[g] = lane_base<COMPACT>(g, lane);
  // byte j of N[r] holds columns 8j + r and 8j + 4 + r: j < 2 is the first
  // half of the word column (columns 0-15), j >= 2 the second
  __half2 hacc[2][R][NT];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int g = 0; g < R; ++g)
#pragma unroll
      for (int tk = 0; tk < NT; ++tk) hacc[hf][g][tk] = __float2half2_rn(0.f);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    uint4 xv[NT];
#pragma unroll
    for (int tk = 0; tk < NT; ++tk) xv[tk] = lds128(xa + tk * kRecBytes + r * 16);
#pragma unroll
    for (int g = 0; g < R; ++g) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 w2 =
            *reinterpret_cast<const __half2*>(g_dsmem + lut_offset<COMPACT>(nb[g][r], lb[g], j));
#pragma unroll
        for (int tk = 0; tk < NT; ++tk) {
          const uint32_t xw = j == 0 ? xv[tk].x : j == 1 ? xv[tk].y : j == 2 ? xv[tk].z : xv[tk].w;
          hacc[j >> 1][g][tk] = __hfma2(w2, *reinterpret_cast<const __half2*>(&xw), hacc[j >> 1][g][tk]);
        }
      }
    }
  }
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) {
    const float2 sc = *reinterpret_cast<const float2*>(g_dsmem + xa + tk * kRecBytes + 64);
#pragma unroll
    for (int g = 0; g < R; ++g) {
      acc[g][tk] = __ffma2_rn(__half22float2(hacc[0][g][tk]), make_float2(sc.x, sc.x), acc[g][tk]);
      acc[g][tk] = __ffma2_rn(__half22float2(hacc[1][g][tk]), make_float2(sc.y, sc.y), acc[g][tk]);
    }
  }
}

template <int Q, int R, int NT, bool COMPACT>
__device__ __forceinline__ void compute_column(uint32_t stage, int lane, const BitConsts& bc,
                                               float2 (&acc)[R][NT]) {
  if constexpr (Form<Q>::kPair) compute_column_pairs<Q, R, NT, COMPACT>(stage, lane, bc, acc);
  else compute_column_bytes<Q, R, NT, COMPACT>(stage, lane, bc, acc);
}

// Start the copies of the warp's first kStages - 1 word columns (one commit
// group each), so that their latency can overlap other set-up work.
template <int Q, int R, int NT>
__device__ __forceinline__ void ring_prime(const uint32_t* planes, long long plane_stride,
                                           long long N, const PassRows<R>& pr, int kw_lo,
                                           int kw_hi, const char* const (&xs)[NT], int nt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = kw_hi - kw_lo;
  if (n <= 0) return;
  const uint32_t ring_s = smem_u32(g_dsmem) + kOffRing + warp * (kStages * kStageBytes);
  const CopyPlan<Q, R, NT> plan = make_copy_plan<Q, R, NT>(plane_stride, pr, xs, nt, lane);
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < n) issue_column<Q, R, NT>(ring_s + i * kStageBytes, planes, N, plan, kw_lo + i, lane);
    cp_async_commit();
  }
}

// Partial dot products of this lane's rows over the warp's word columns
// [kw_lo, kw_hi), streamed through the warp's kStages-deep cp.async ring
// (whose first columns were already started when `primed`).
template <int Q, int R, int NT, bool COMPACT>
__device__ __forceinline__ void rows_dot(const uint32_t* planes, long long plane_stride, long long N,
                                         const PassRows<R>& pr, int kw_lo, int kw_hi,
                                         const char* const (&xs)[NT], int nt, const SmemPtrs& s,
                                         const BitConsts& bc, float2 (&acc)[R][NT], bool primed) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int g = 0; g < R; ++g)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[g][t] = make_float2(0.f, 0.f);
  const int n = kw_hi - kw_lo;
  if (n <= 0) return;
  const uint32_t ring = kOffRing + warp * (kStages * kStageBytes);   // offset in g_dsmem
  const uint32_t ring_s = smem_u32(g_dsmem) + ring;
  const CopyPlan<Q, R, NT> plan = make_copy_plan<Q, R, NT>(plane_stride, pr, xs, nt, lane);
  if (!primed) ring_prime<Q, R, NT>(planes, plane_stride, N, pr, kw_lo, kw_hi, xs, nt);
  for (int i = 0; i < n; ++i) {
    const int pf = i + kStages - 1;
    if (pf < n)
      issue_column<Q, R, NT>(ring_s + (pf % kStages) * kStageBytes, planes, N, plan, kw_lo + pf,
                             lane);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    compute_column<Q, R, NT, COMPACT>(ring + (i % kStages) * kStageBytes, lane, bc, acc);
    __syncwarp();
  }
}

__device__ __forceinline__ void warp_range(int KW, int& lo, int& hi) {
  const int warp = threadIdx.x >> 5;
  lo = (warp * KW) / kWarps;
  hi = ((warp + 1) * KW) / kWarps;
}

// This warp's word columns of K part kh of KS (the parts split [0, KW) at KW/KS).
template <int KS>
__device__ __forceinline__ void warp_range_part(int KW, int kh, int& lo, int& hi) {
  if constexpr (KS == 1) {
    warp_range(KW, lo, hi);
  } else {
    const int warp = threadIdx.x >> 5;
    const int k0 = kh * (KW / KS), kc = (kh == KS - 1) ? KW - k0 : KW / KS;
    lo = k0 + (warp * kc) / kWarps;
    hi = k0 + ((warp + 1) * kc) / kWarps;
  }
}


// Spin bound of the down kernel's wait for an expert's gate_up tiles; the
// wait backs off with a short sleep, so the bound is well over a second.
constexpr uint32_t kReadySpinLimit = 1u << 23;

// Largest down-block K (= I) whose tiles start per expert (see above).
constexpr int kEarlyDownMaxI = 8192;

__device__ __forceinline__ int load_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Thread 0 of a down CTA: wait until `need` gate_up tiles of the expert have
// released their h rows.  `seen` is a poll issued earlier (relaxed, so that
// it overlaps other loads); the closing fence makes the wait an acquire.
// Gives up after kReadySpinLimit polls and latches PW_ERR_TIMEOUT (the tile
// then runs on whatever h holds).
__device__ __forceinline__ void wait_gate_up(const int* done, int seen, int need,
                                             int32_t* status, uint32_t limit = kReadySpinLimit) {
  for (uint32_t i = 0; seen < need; ++i) {
    if (i == limit) {
      latch_status(status, PW_ERR_TIMEOUT);
      break;
    }
    __nanosleep(128);
    seen = load_relaxed(done);
  }
  __threadfence();
}

// A counter that nothing ever increments: the bounded-wait check below waits
// on it so that the wait must run out.
__device__ int g_never_released = 0;

// Failure-detection check: the down kernel's wait for an expert's gate_up
// tiles, run by one thread on a counter nobody releases, with `limit` polls.
// It must give up, latch PW_ERR_TIMEOUT and return.
__global__ void wait_check_kernel(int32_t* status, uint32_t limit) {
  if (threadIdx.x == 0) wait_gate_up(&g_never_released, load_relaxed(&g_never_released), 1, status, limit);
}

// ---------------------------------------------------------------- gate_up

// Activation rows of one token group, as byte pointers to word column 0 of
// each token's row in the form of bitwidth Q.
template <int Q, int NT>
__device__ __forceinline__ void gateup_xs(const LayerArgs& a, const DecodeWs& w,
                                          const ExpertWork& ex, const SlotInfo& ent, int g0, int nt,
                                          const char* (&xs)[NT]) {
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) {
    const long long row = g0 == 0 ? ent.rows[tk] : w.perm[ex.off + g0 + min(tk, nt - 1)] / a.k;
    xs[tk] = Form<Q>::kPair ? w.xp + row * (a.H / 32) * kRecBytes
                            : reinterpret_cast<const char*>(w.xs + row * a.H);
  }
}

template <int Q, int R, int NT>
__device__ void gateup_prime(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                             const SlotInfo& ent, const PassRows<R>& pr, int g0, int nt) {
  const int KW = a.H / 32;
  const long long N = 2LL * a.I;
  int lo, hi;
  warp_range(KW, lo, hi);
  const char* xs[NT];
  gateup_xs<Q, NT>(a, w, ex, ent, g0, nt, xs);
  ring_prime<Q, R, NT>(ent.planes, N * KW, N, pr, lo, hi, xs, nt);
}

// Writes one token's h values of a pass (lane L holds column hcol0 + L for
// L < width) in the form the expert's down block reads.  The fp16 form's
// scale belongs to a half of the group of 32 columns (16 columns), which a
// compact pass (width 16) covers alone and a paired pass (width 32) covers
// with lanes 0-15 and 16-31.
__device__ __forceinline__ void store_h(const LayerArgs& a, const DecodeWs& w, int pos, int hcol0,
                                        int width, int lane, float h, bool fp16_form) {
  const int col = hcol0 + lane;
  if (!fp16_form) {
    float* hs_row = w.hs + static_cast<long long>(pos) * a.I;
    if (lane < width) hs_row[(col & ~31) + byte_form_position(col & 31)] = h;
    return;
  }
  char* rec = w.hp + (static_cast<long long>(pos) * (a.I / 32) + (hcol0 >> 5)) * kRecBytes;
  float m = lane < width ? fabsf(h) : 0.f;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  const int e = group_exponent(m);
  if (lane < width) {
    reinterpret_cast<__half*>(rec)[nibble_form_position(col & 31)] = __float2half_rn(h * exp2i(-e));
    if ((lane & 15) == 0)
      *reinterpret_cast<float*>(rec + 64 + 4 * ((col >> 4) & 1)) = exp2i(e);
  }
}

template <int Q, int R, bool COMPACT, int NT>
__device__ void gateup_group(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                             const SlotInfo& ent, const PassRows<R>& pr, int hcol0, int g0,
                             int nt, const SmemPtrs& s, const BitConsts& bc, bool primed,
                             int* claim_counter) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KW = a.H / 32;
  const long long N = 2LL * a.I;
  int lo, hi;
  warp_range(KW, lo, hi);
  PW_DTRACE_MARK(tr_cols);
  const char* xs[NT];
  gateup_xs<Q, NT>(a, w, ex, ent, g0, nt, xs);
  float2 acc[R][NT];
  rows_dot<Q, R, NT, COMPACT>(ent.planes, N * KW, N, pr, lo, hi, xs, nt, s, bc, acc, primed);
  // the tile's last group claims the CTA's next tile from the last warp,
  // which the reduction leaves idle (kTG < kWarps), so that no reducing warp
  // waits for the atomic; its round trip overlaps the partial-sum stores and
  // the reduction
  int claim = 0;
  if (claim_counter && threadIdx.x == 32 * (kWarps - 1)) claim = atomicAdd(claim_counter, 1);
#pragma unroll
  for (int tk = 0; tk < NT; ++tk)
#pragma unroll
    for (int g = 0; g < R; ++g)
      s.red[((warp * kTG + tk) * 2 + g) * 32 + lane] = acc[g][tk].x + acc[g][tk].y;
  __syncthreads();
  PW_DTRACE_ADD(s, 4, tr_cols);
  PW_DTRACE_MARK(tr_red);
  if (threadIdx.x < 32 * nt) {   // warp tk finishes token tk
    const int tk = threadIdx.x >> 5;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
      v0 += s.red[((ww * kTG + tk) * 2 + 0) * 32 + lane];
      if (R == 2) v1 += s.red[((ww * kTG + tk) * 2 + 1) * 32 + lane];
    }
    if (R == 1) v1 = __shfl_xor_sync(kFull, v0, 16);
    const int width = (R == 2) ? 32 : 16;
    const float h = lane < width ? v0 / (1.f + expf(-v0)) * v1 : 0.f;
    store_h(a, w, ex.off + g0 + tk, hcol0, width, lane, h, ent.q_other <= 4);
  } else if (claim_counter && threadIdx.x == 32 * (kWarps - 1)) {
    s.misc[2] = claim;
  }
  __syncthreads();
  PW_DTRACE_ADD(s, 5, tr_red);
}

template <int Q, int R, bool COMPACT>
__device__ void gateup_pass(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                            const SlotInfo& ent, const PassRows<R>& pr, int hcol0,
                            const SmemPtrs& s, const BitConsts& bc, int* claim_counter) {
  PW_DTRACE_MARK(tr_setup);
  __syncthreads();  // the previous pass is done with the LUT region and the rings
  // the LUT loads go out first, then the first token group's first columns
  // (whose activation rows need one more dependent load), so that both
  // round trips overlap
  PassLut<Q, R> pl;
  pass_lut_fetch<Q, R>(ent.lut, pr, pl);
  const int nt0 = min(kTG, ex.ne);
  if (nt0 == 1) gateup_prime<Q, R, 1>(a, w, ex, ent, pr, 0, nt0);
  else gateup_prime<Q, R, kTG>(a, w, ex, ent, pr, 0, nt0);
  PW_DTRACE_ADD(s, 7, tr_setup);
  PW_DTRACE_MARK(tr_build);
  pass_lut_store<Q, R, COMPACT>(pl, a.status);
  PW_DTRACE_ADD(s, 8, tr_build);
  PW_DTRACE_MARK(tr_bar);
  __syncthreads();
  PW_DTRACE_ADD(s, 9, tr_bar);
  PW_DTRACE_ADD(s, 3, tr_setup);
  // token groups of one token take the one-token code; 2-4 tokens the kTG
  // code, with the missing tokens zero-filled (fewer code variants keep the
  // instruction cache warm)
  for (int g0 = 0; g0 < ex.ne; g0 += kTG) {
    const int nt = min(kTG, ex.ne - g0);
    const bool primed = (g0 == 0);
    int* cc = (g0 + kTG >= ex.ne) ? claim_counter : nullptr;
    if (nt == 1) gateup_group<Q, R, COMPACT, 1>(a, w, ex, ent, pr, hcol0, g0, nt, s, bc, primed, cc);
    else gateup_group<Q, R, COMPACT, kTG>(a, w, ex, ent, pr, hcol0, g0, nt, s, bc, primed, cc);
  }
}

// One row per lane for the bitwidths whose tables fill the LUT region.
template <int Q>
constexpr bool compact_q() { return Q == 4 || Q == 8; }

template <int Q>
__device__ void gateup_tile(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                            const SlotInfo& ent, int i0, const SmemPtrs& s,
                            const BitConsts& bc, int* claim_counter) {
  if constexpr (compact_q<Q>()) {
    // two passes of 16 h columns: lanes 0-15 gate rows, lanes 16-31 up rows
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int i = i0 + 16 * half;
      PassRows<1> pr;
      pr.seg[0][0] = i;
      pr.seg[0][1] = a.I + i;
      gateup_pass<Q, 1, true>(a, w, ex, ent, pr, i, s, bc, half ? claim_counter : nullptr);
    }
  } else {
    PassRows<2> pr;
    pr.seg[0][0] = i0;
    pr.seg[0][1] = i0 + 16;
    pr.seg[1][0] = a.I + i0;
    pr.seg[1][1] = a.I + i0 + 16;
    gateup_pass<Q, 2, false>(a, w, ex, ent, pr, i0, s, bc, claim_counter);
  }
}

__global__ void __launch_bounds__(kThreads, 2) decode_gateup_kernel(const LayerArgs a,
                                                                    const DecodeWs w,
                                                                    const BitConsts bc) {
  const SmemPtrs s = carve(g_dsmem);
  grid_dependency_wait();      // routing and fp32 hidden states are ready
  allow_dependent_launch();    // the down kernel may start loading as CTAs retire
  const int tpe = a.I / kPairsPerTile;
  const int total = w.ctl[0] * tpe;
  int* const counter = &w.ctl[1];
  // Thread 0 releases a finished tile's h rows to the down kernel one tile
  // late: by the next tile's descriptor load the stores have long landed,
  // so the fence costs little.  The barriers since the tile's last h store
  // order every thread's stores before thread 0's fence.
  int pending = -1;
#ifdef PW_TRACE
  int tr_tiles = 0;
#endif
  // A CTA's first tile is its block index; each tile claims the next one
  // from the counter (offset by the grid size) and leaves it in misc[2].
  for (int t = blockIdx.x; t < total;) {
    PW_DTRACE_TILE_BEGIN(s, tr_tiles++, tr_desc);
    const int slot = t / tpe, x = t - slot * tpe;
    const SlotInfo si = w.routed_gu[slot];
    if (threadIdx.x == 0 && pending >= 0) {
      __threadfence();
      atomicAdd(&w.gu_done[pending], 1);
      pending = -1;
    }
    if (si.err || si.ne <= 0) {   // (a routed expert always holds a pair)
      if (threadIdx.x == 0) {
        if (si.err > 0 && x == 0) latch_status(a.status, si.err);   // -1: reported elsewhere
        s.misc[2] = atomicAdd(counter, 1);
      }
      __syncthreads();
    } else {
      PW_DTRACE_ADD(s, 2, tr_desc);   // the branch above waited for the descriptor
      const ExpertWork ex{si.e, si.off, si.ne};
      switch (si.q) {
        case 3: gateup_tile<3>(a, w, ex, si, x * kPairsPerTile, s, bc, counter); break;
        case 4: gateup_tile<4>(a, w, ex, si, x * kPairsPerTile, s, bc, counter); break;
        case 5: gateup_tile<5>(a, w, ex, si, x * kPairsPerTile, s, bc, counter); break;
        case 6: gateup_tile<6>(a, w, ex, si, x * kPairsPerTile, s, bc, counter); break;
        default: gateup_tile<8>(a, w, ex, si, x * kPairsPerTile, s, bc, counter); break;
      }
      if (a.I <= kEarlyDownMaxI) pending = si.off;   // the down tiles wait per token group
      PW_DTRACE_TILE_END(s, si.q, si.ne);
    }
    // claims only grow, so a tile id that does not advance ends the loop
    const int next = static_cast<int>(gridDim.x) + s.misc[2];
    t = next > t ? next : total;
    __syncthreads();   // every thread has read the claim before it is overwritten
  }
  if (threadIdx.x == 0 && pending >= 0) {
    __threadfence();
    atomicAdd(&w.gu_done[pending], 1);
  }
  PW_DTRACE_EXIT();
}

// ---------------------------------------------------------------- down

template <int Q, int NT>
__device__ __forceinline__ void down_xs(const LayerArgs& a, const DecodeWs& w,
                                        const ExpertWork& ex, int g0, int nt,
                                        const char* (&xs)[NT]) {
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) {
    const long long pos = ex.off + g0 + min(tk, nt - 1);
    xs[tk] = Form<Q>::kPair ? w.hp + pos * (a.I / 32) * kRecBytes
                            : reinterpret_cast<const char*>(w.hs + pos * a.I);
  }
}

template <int Q, int R, int NT, int KS>
__device__ void down_prime(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                           const SlotInfo& ent, const PassRows<R>& pr, int g0, int nt, int kh) {
  const int KW = a.I / 32;
  const long long N = a.H;
  int lo, hi;
  warp_range_part<KS>(KW, kh, lo, hi);
  const char* xs[NT];
  down_xs<Q, NT>(a, w, ex, g0, nt, xs);
  ring_prime<Q, R, NT>(ent.planes, N * KW, N, pr, lo, hi, xs, nt);
}

template <int Q, int R, bool COMPACT, int NT, int KS>
__device__ void down_group(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                           const SlotInfo& ent, const PassRows<R>& pr, int g0, int nt,
                           const SmemPtrs& s, const BitConsts& bc, bool primed, int kh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KW = a.I / 32;
  const long long N = a.H;
  int lo, hi;
  warp_range_part<KS>(KW, kh, lo, hi);
  const char* xs[NT];
  down_xs<Q, NT>(a, w, ex, g0, nt, xs);
  float2 acc[R][NT];
  rows_dot<Q, R, NT, COMPACT>(ent.planes, N * KW, N, pr, lo, hi, xs, nt, s, bc, acc, primed);
  // thread i < 32*R*nt (at most kThreads) writes row slot (i/32)%R of token
  // (i/32)/R; its pair id is loaded before the partial sums meet
  const int i = threadIdx.x;
  const bool writer = i < 32 * R * nt;
  const int pair = writer ? w.perm[ex.off + g0 + (i >> 5) / R] : 0;
#pragma unroll
  for (int tk = 0; tk < NT; ++tk)
#pragma unroll
    for (int g = 0; g < R; ++g)
      s.red[((warp * kTG + tk) * 2 + g) * 32 + lane] = acc[g][tk].x + acc[g][tk].y;
  __syncthreads();
  if (writer) {
    const int g = (i >> 5) % R, tk = (i >> 5) / R;
    float y = 0.f;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) y += s.red[((ww * kTG + tk) * 2 + g) * 32 + lane];
    const int row = seg_base<R>(pr, g, lane >> 4) + (lane & 15);
    ((KS == 2 && kh) ? w.y2 : w.y)[static_cast<long long>(pair) * a.H + row] = y;
  }
  __syncthreads();
}

template <int Q, int R, bool COMPACT, int KS>
__device__ void down_pass(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                          const SlotInfo& ent, const PassRows<R>& pr, const SmemPtrs& s,
                          const BitConsts& bc, int kh) {
  __syncthreads();
  // the expert's h rows are complete once all of its gate_up tiles released
  // them: thread 0 polls (the first poll overlaps the LUT load) and acquires,
  // and the barrier extends that to the CTA
  const bool early = a.I <= kEarlyDownMaxI;
  const int seen = (early && threadIdx.x == 0) ? load_relaxed(w.gu_done + ex.off) : 0;
  {  // the LUT does not depend on h
    PassLut<Q, R> pl;
    pass_lut_fetch<Q, R>(ent.lut, pr, pl);
    pass_lut_store<Q, R, COMPACT>(pl, a.status);
  }
  if (!early) grid_dependency_wait();   // the whole gate_up grid is done
  else if (threadIdx.x == 0) wait_gate_up(w.gu_done + ex.off, seen, a.I / kPairsPerTile, a.status);
  __syncthreads();
  const int nt0 = min(kTG, ex.ne);
  if (nt0 == 1) down_prime<Q, R, 1, KS>(a, w, ex, ent, pr, 0, nt0, kh);
  else down_prime<Q, R, kTG, KS>(a, w, ex, ent, pr, 0, nt0, kh);
  for (int g0 = 0; g0 < ex.ne; g0 += kTG) {
    const int nt = min(kTG, ex.ne - g0);
    const bool primed = (g0 == 0);
    if (nt == 1) down_group<Q, R, COMPACT, 1, KS>(a, w, ex, ent, pr, g0, nt, s, bc, primed, kh);
    else down_group<Q, R, COMPACT, kTG, KS>(a, w, ex, ent, pr, g0, nt, s, bc, primed, kh);
  }
}

// A down tile of `rows` (64, or 32 on a ragged last tile) rows from n0.
template <int Q, int KS>
__device__ void down_tile(const LayerArgs& a, const DecodeWs& w, const ExpertWork& ex,
                          const SlotInfo& ent, int n0, int rows, const SmemPtrs& s,
                          const BitConsts& bc, int kh) {
  if (compact_q<Q>() || rows == 32) {
#pragma unroll 1
    for (int grp = 0; grp < rows / 32; ++grp) {
      PassRows<1> pr;
      pr.seg[0][0] = n0 + 32 * grp;
      pr.seg[0][1] = n0 + 32 * grp + 16;
      if constexpr (compact_q<Q>()) down_pass<Q, 1, true, KS>(a, w, ex, ent, pr, s, bc, kh);
      else down_pass<Q, 1, false, KS>(a, w, ex, ent, pr, s, bc, kh);
    }
  } else {
    PassRows<2> pr;
    pr.seg[0][0] = n0;
    pr.seg[0][1] = n0 + 16;
    pr.seg[1][0] = n0 + 32;
    pr.seg[1][1] = n0 + 48;
    down_pass<Q, 2, false, KS>(a, w, ex, ent, pr, s, bc, kh);
  }
}

// out[t][c] = sum_j w_tj * y[t k + j][c] over the token's valid pairs, in j
// order, for every token t and columns c in [n0, n0 + cols) (cols a multiple
// of 4): four columns per work item, items i0, i0 + stride, ...
template <int KS>
__device__ void combine_columns(const LayerArgs& a, const DecodeWs& w, int n0, int cols, int i0,
                                int stride) {
  const int c4 = cols / 4;
  const int items = a.T * c4;
  for (int i = i0; i < items; i += stride) {
    const int tt = i / c4, c = n0 + 4 * (i - tt * c4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int j = 0; j < a.k; ++j) {
      const int p = tt * a.k + j;
      const int e = a.topk_ids[p];
      if (e < 0 || e >= a.E) continue;
      const float wt = a.topk_weights[p];
      float4 v = __ldcg(reinterpret_cast<const float4*>(w.y + static_cast<long long>(p) * a.H + c));
      if constexpr (KS == 2) {   // the down tiles' second K half
        const float4 v2 =
            __ldcg(reinterpret_cast<const float4*>(w.y2 + static_cast<long long>(p) * a.H + c));
        v.x += v2.x;
        v.y += v2.y;
        v.z += v2.z;
        v.w += v2.w;
      }
      acc.x = fmaf(wt, v.x, acc.x);
      acc.y = fmaf(wt, v.y, acc.y);
      acc.z = fmaf(wt, v.z, acc.z);
      acc.w = fmaf(wt, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(a.out + static_cast<long long>(tt) * a.H + c) = acc;
  }
}

// KS: K parts per 64-row range (1, or 2 for long down blocks in calls with
// few down tiles; the second part's partial sums go to y2).
template <int KS>
__global__ void __launch_bounds__(kThreads, 2) decode_down_kernel(const LayerArgs a,
                                                                  const DecodeWs w,
                                                                  const BitConsts bc) {
  const SmemPtrs s = carve(g_dsmem);
  // with SM slots to spare, the next call's prep (launched early in that
  // case) may become resident now and wait for this grid to finish
  if (w.early_next) allow_dependent_launch();
  // Routing (from the prep launch, which finished before the gate_up
  // kernel allowed this launch) is readable now; h only after the wait.
  const int n_routed = w.ctl[0];
  if (n_routed == 0) {
    // every routed expert went to the GEMM kernels (or none was routed):
    // only the combine is left
    grid_dependency_wait();
    combine_columns<1>(a, w, 0, a.H, static_cast<int>(blockIdx.x) * kThreads + threadIdx.x,
                       static_cast<int>(gridDim.x) * kThreads);
    return;
  }
  const int tpe = (a.H + kDownRows - 1) / kDownRows;
  // a tile is (slot, 64-row range, K part); the K parts of a range are
  // neighbouring tiles
  constexpr int ks = KS;
  const int total = n_routed * tpe * ks;
  // A CTA's first tile is its block index; each tile claims the next one
  // from the counter (offset by the grid size) together with its arrival.
  for (int t = blockIdx.x; t < total;) {
    const int slot = t / (tpe * ks), rem = t - slot * (tpe * ks);
    const int x = rem / ks, kh = rem - x * ks;
    const SlotInfo si = w.routed_dn[slot];
    const ExpertWork ex{si.e, si.off, si.ne};
    const int n0 = x * kDownRows;
    const int rows = min(kDownRows, a.H - n0);   // 64, or 32 on a ragged last range
    if (si.err) {
      // this expert contributes zero; gate_up skipped it (h is not valid)
      if (x == 0 && kh == 0 && threadIdx.x == 0 && si.err > 0) latch_status(a.status, si.err);
      float* const yk = (KS == 2 && kh) ? w.y2 : w.y;
      for (int i = threadIdx.x; i < ex.ne * rows; i += kThreads)
        yk[static_cast<long long>(w.perm[ex.off + i / rows]) * a.H + n0 + (i % rows)] = 0.f;
    } else {
      switch (si.q) {
        case 3: down_tile<3, KS>(a, w, ex, si, n0, rows, s, bc, kh); break;
        case 4: down_tile<4, KS>(a, w, ex, si, n0, rows, s, bc, kh); break;
        case 5: down_tile<5, KS>(a, w, ex, si, n0, rows, s, bc, kh); break;
        case 6: down_tile<6, KS>(a, w, ex, si, n0, rows, s, bc, kh); break;
        default: down_tile<8, KS>(a, w, ex, si, n0, rows, s, bc, kh); break;
      }
    }
    // Arrival: the last routed expert to finish this row range combines it.
    // The barrier orders every thread's y stores before thread 0's fence and
    // arrival (the release); the claim of the next tile shares the round trip.
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int arrived = atomicAdd(&w.arrive[x], 1);
      const int claim = atomicAdd(&w.ctl[2], 1);
      s.misc[1] = (arrived == n_routed * ks - 1);
      s.misc[2] = claim;
    }
    __syncthreads();
    if (s.misc[1]) {
      __threadfence();
      combine_columns<KS>(a, w, n0, rows, threadIdx.x, kThreads);
    }
    const int next = static_cast<int>(gridDim.x) + s.misc[2];
    t = next > t ? next : total;
    __syncthreads();   // every thread has read the flags before they are overwritten
  }
}

// ---------------------------------------------------------------- prep

__device__ __forceinline__ int q_class(int q) {
  return q == 8 ? 0 : q == 6 ? 1 : q == 5 ? 2 : q == 4 ? 3 : q == 3 ? 4 : 5;
}

// CTA 0: stable grouping of pairs by expert (offsets, perm), routed-expert
// lists ordered by bitwidth class (largest first; order inside a class does
// not matter), counters reset.  Other CTAs: hidden -> both activation forms
// (fp32, and fp16 records with their group scales) and out = 0.
__global__ void __launch_bounds__(kPrepThreads) decode_prep_kernel(const LayerArgs a,
                                                                   const DecodeWs w) {
  // when launched early (programmatic dependent launch), nothing of the
  // previous kernel on the stream (which may be an earlier call still reading
  // this workspace and writing `out`) is touched before it completes
  if (w.early_next) grid_dependency_wait();
  allow_dependent_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (blockIdx.x != 0) {
    // unit i = 4 columns; the 8 units of a group of 32 columns are 8
    // consecutive lanes (H is a multiple of 32), and every lane of a warp
    // runs every iteration, so a half's maximum (4 units) is a 2-step shuffle
    const long long n4 = static_cast<long long>(a.T) * a.H / 4;
    const long long stride = static_cast<long long>(gridDim.x - 1) * kPrepThreads;
    for (long long base = static_cast<long long>(blockIdx.x - 1) * kPrepThreads; base < n4;
         base += stride) {
      const long long i = base + tid;
      const bool valid = i < n4;
      const uint2 raw = valid ? __ldg(reinterpret_cast<const uint2*>(a.hidden) + i) : make_uint2(0, 0);
      const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                          __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
      float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));   // a half: 16 columns
      if (valid) {
        const long long grp = i >> 3;          // (token, group of 32 columns)
        const int u = static_cast<int>(i & 7);  // columns 4u .. 4u+3 of the group
        float* xs_g = w.xs + grp * 32;
        char* rec = w.xp + grp * kRecBytes;
        const int e = group_exponent(m);
        const float down = exp2i(-e);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xs_g[byte_form_position(4 * u + j)] = v[j];
          reinterpret_cast<__half*>(rec)[nibble_form_position(4 * u + j)] =
              __float2half_rn(v[j] * down);
        }
        if ((u & 3) == 0) *reinterpret_cast<float*>(rec + 64 + 4 * (u >> 2)) = exp2i(e);
        reinterpret_cast<float4*>(a.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }
  extern __shared__ int psm[];
  const int E = a.E, P = a.T * a.k;
  if (a.logits != nullptr) {
    // fused routing: the warps route the tokens into topk_ids / topk_weights
    // (the caller's buffers, by-products of the call) before the grouping
    for (int t = warp; t < a.T; t += kPrepWarps)
      route_token_warp(a.logits + static_cast<long long>(t) * E, E, a.k,
                       a.route_ids + static_cast<long long>(t) * a.k,
                       a.route_wts + static_cast<long long>(t) * a.k);
    __syncthreads();   // the routed ids are visible to the whole CTA
  }
  int* count = psm;                 // [E]
  int* base = count + E;            // [E]
  int* wcnt = base + E;             // [kPrepWarps][E]
  float* wsum = reinterpret_cast<float*>(wcnt + kPrepWarps * E);   // [E] routing mass
  const bool stats = a.stats_counts != nullptr;
  __shared__ int s_warp_sum[kPrepWarps];
  __shared__ int s_bucket[2][8];
  // the page-table entries of this thread's first expert load now, so that
  // their round trip overlaps the pair counting
  pw_block_entry t_gu = {}, t_dn = {};
  if (tid < E) {
    t_gu = a.table[2 * tid];
    t_dn = a.table[2 * tid + 1];
  }
  for (int e = tid; e < E; e += kPrepThreads) {
    count[e] = 0;
    wsum[e] = 0.f;
  }
  for (int p = tid; p < P; p += kPrepThreads) w.gu_done[p] = 0;
  for (int i = tid; i < kPrepWarps * E; i += kPrepThreads) wcnt[i] = 0;
  if (tid < 16) (&s_bucket[0][0])[tid] = 0;
  for (int i = tid; i < (a.H + 31) / 32; i += kPrepThreads) w.arrive[i] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += kPrepThreads) {
    const int e = a.topk_ids[p];
    if (e >= 0 && e < E) {
      atomicAdd(&count[e], 1);
      if (stats) atomicAdd(&wsum[e], a.topk_weights[p]);
    } else {
      latch_status(a.status, PW_ERR_BAD_EXPERT_ID);
    }
  }
  __syncthreads();
  if (stats) {   // routing statistics, a by-product of the grouping
    for (int e = tid; e < E; e += kPrepThreads) {
      if (count[e] > 0) {
        atomicAdd(&a.stats_counts[e], count[e]);
        atomicAdd(&a.stats_mass[e], wsum[e]);
      }
    }
  }
  // exclusive scan of count -> base / offsets
  const int per = (E + kPrepThreads - 1) / kPrepThreads;
  const int lo = min(E, tid * per), hi = min(E, lo + per);
  int run = 0;
  for (int e = lo; e < hi; ++e) run += count[e];
  int incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp_sum[warp] = incl;
  __syncthreads();
  int before = incl - run;
  for (int ww = 0; ww < warp; ++ww) before += s_warp_sum[ww];
  for (int e = lo; e < hi; ++e) {
    base[e] = before;
    w.offsets[e] = before;
    before += count[e];
  }
  if (tid == kPrepThreads - 1) {
    int total = 0;
    for (int ww = 0; ww < kPrepWarps; ++ww) total += s_warp_sum[ww];
    w.offsets[E] = total;
  }
  // routed experts by bitwidth class (experts the GEMM kernels take are left out)
  const int heavy_min = w.heavy_min > 0 ? w.heavy_min : INT_MAX;
  // one slot per (expert, group of up to kTG pairs): an expert's groups are
  // independent tiles, so that a heavily routed expert spreads over many
  // CTAs instead of looping over its groups inside each tile
  for (int e = tid; e < E; e += kPrepThreads) {
    if (count[e] > 0 && count[e] < heavy_min) {
      const int ng = (count[e] + kTG - 1) / kTG;
      atomicAdd(&s_bucket[0][q_class(e == tid ? t_gu.q : a.table[2 * e].q)], ng);
      atomicAdd(&s_bucket[1][q_class(e == tid ? t_dn.q : a.table[2 * e + 1].q)], ng);
    }
  }
  __syncthreads();
  if (tid < 2) {
    int acc = 0;
    for (int c = 0; c < 6; ++c) {
      const int n = s_bucket[tid][c];
      s_bucket[tid][c] = acc;
      acc += n;
    }
    if (tid == 0) {
      w.ctl[0] = acc;
      w.ctl[1] = 0;
      w.ctl[2] = 0;
    }
  }
  __syncthreads();
  // stable placement: rank among same-expert lanes (match), earlier warps of
  // the chunk (per-warp counts) and earlier chunks (running base)
  for (int c0 = 0; c0 < P; c0 += kPrepThreads) {
    const int p = c0 + tid;
    const int e = (p < P) ? a.topk_ids[p] : -1;
    const bool valid = (e >= 0 && e < E);
    const unsigned peers = __match_any_sync(kFull, valid ? e : -1);
    const unsigned lower = peers & ((1u << lane) - 1u);
    if (valid && lower == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int pos = base[e] + __popc(lower);
      for (int ww = 0; ww < warp; ++ww) pos += wcnt[ww * E + e];
      w.perm[pos] = p;
    }
    __syncthreads();
    for (int x = tid; x < E; x += kPrepThreads) {
      int add = 0;
      for (int ww = 0; ww < kPrepWarps; ++ww) {
        add += wcnt[ww * E + x];
        wcnt[ww * E + x] = 0;
      }
      base[x] += add;
    }
    __syncthreads();
  }
  // slot descriptors, once the placement is done (perm is readable by the
  // whole CTA after the loop's last barrier; base[e] has moved past e's
  // pairs)
  for (int e = tid; e < E; e += kPrepThreads) {
    if (count[e] > 0 && count[e] < heavy_min) {
      const pw_block_entry gu = e == tid ? t_gu : a.table[2 * e];
      const pw_block_entry dn = e == tid ? t_dn : a.table[2 * e + 1];
      const bool gu_ok = gu.state == PW_PAGE_GPU && supported_q(gu.q);
      const bool dn_ok = dn.state == PW_PAGE_GPU && supported_q(dn.q);
      const int first = base[e] - count[e];
      const int gu_err = gu_ok ? PW_OK
                               : (gu.state != PW_PAGE_GPU ? PW_ERR_PAGE_NOT_RESIDENT : PW_ERR_UNSUPPORTED_Q);
      // down tiles of an expert whose gate_up block cannot run write zeros
      // (their h is not valid); the error was latched by the gate_up tiles
      const int dn_err = !gu_ok ? -1
                         : dn_ok ? PW_OK
                                 : (dn.state != PW_PAGE_GPU ? PW_ERR_PAGE_NOT_RESIDENT : PW_ERR_UNSUPPORTED_Q);
      for (int g0 = 0; g0 < count[e]; g0 += kTG) {
        SlotInfo si;
        si.e = e;
        si.off = first + g0;
        si.ne = min(kTG, count[e] - g0);
#pragma unroll
        for (int i = 0; i < 4; ++i) si.rows[i] = w.perm[si.off + min(i, si.ne - 1)] / a.k;
        si.q_other = dn.q;
        si.q = gu.q;
        si.planes = gu.planes;
        si.lut = gu.lut;
        // only the expert's first group reports its error
        si.err = g0 == 0 ? gu_err : (gu_err ? -1 : PW_OK);
        w.routed_gu[atomicAdd(&s_bucket[0][q_class(gu.q)], 1)] = si;
        si.q = dn.q;
        si.q_other = gu.q;
        si.planes = dn.planes;
        si.lut = dn.lut;
        si.err = g0 == 0 ? dn_err : (dn_err > 0 ? -1 : dn_err);
        w.routed_dn[atomicAdd(&s_bucket[1][q_class(dn.q)], 1)] = si;
      }
    }
  }
}

}  // namespace

cudaError_t launch_wait_check_decode(int32_t* status, uint32_t polls, cudaStream_t s) {
  wait_check_kernel<<<1, 32, 0, s>>>(status, polls);
  return cudaGetLastError();
}

namespace {
// The >48 KB shared-memory opt-in of the decode kernels, set once per device.
cudaError_t configure_decode() {
  cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_down_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_down_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmemBytes));
}
}  // namespace

namespace {

// ---------------------------------------------------------------- checks
//
// The decode kernels' index extraction and table lookups, run on a whole
// block and written back in column order, so that they can be compared bit
// for bit with the format's definition.  The column order of each index
// form is the one the kernels' activation layouts assume.

// One thread per (row n, word column w): the q plane words, the kernels'
// extraction, each index stored at its column.
template <int Q, bool NIBBLES>
__global__ void __launch_bounds__(256) index_check_kernel(const uint32_t* __restrict__ planes, int N,
                                                          int KW, uint8_t* __restrict__ idx,
                                                          const BitConsts bc) {
  const long long total = static_cast<long long>(N) * KW;
  const long long plane = total;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long wcol = i / N, n = i % N;
    uint32_t P[Q];
#pragma unroll
    for (int p = 0; p < Q; ++p) P[p] = planes[p * plane + wcol * N + n];
    uint8_t* row = idx + n * (32LL * KW) + 32 * wcol;
    if constexpr (NIBBLES) {
      uint32_t nb[4];
      planes_to_nibbles<Q>(P, nb, bc);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int m = 0; m < 8; ++m) row[4 * m + r] = static_cast<uint8_t>((nb[r] >> (4 * m)) & 15u);
    } else {
      uint32_t b8[8];
      planes_to_bytes<Q>(P, b8, bc);
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int b = 0; b < 4; ++b) row[8 * b + r] = static_cast<uint8_t>((b8[r] >> (8 * b)) & 255u);
    }
  }
}

// One CTA (kThreads) per pass of rows, as the gate_up / down kernels run it:
// 64 rows in two slots, or 32 rows in one (compact bitwidths, or a ragged
// last 32 rows).  The pass's table is built with the kernels' fetch and
// store, then lane L of a slot looks up its row's indices with the kernels'
// offsets and writes each weight at its column (pair tables give two).
template <int Q, int R, bool COMPACT>
__device__ void dequant_check_pass(const uint32_t* planes, const uint16_t* lut, int N, int KW,
                                   int n0, float* out, const BitConsts& bc, int32_t* status) {
  PassRows<R> pr;
  pr.seg[0][0] = n0;
  pr.seg[0][1] = n0 + 16;
  if (R == 2) {
    pr.seg[R - 1][0] = n0 + 32;
    pr.seg[R - 1][1] = n0 + 48;
  }
  __syncthreads();   // the previous pass is done with the table
  {
    PassLut<Q, R> pl;
    pass_lut_fetch<Q, R>(lut, pr, pl);
    pass_lut_store<Q, R, COMPACT>(pl, status);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long plane = static_cast<long long>(N) * KW;
  for (int wcol = warp; wcol < KW; wcol += kWarps) {
#pragma unroll
    for (int g = 0; g < R; ++g) {
      const int row = seg_base<R>(pr, g, lane >> 4) + (lane & 15);
      uint32_t P[Q];
#pragma unroll
      for (int p = 0; p < Q; ++p) P[p] = planes[p * plane + static_cast<long long>(wcol) * N + row];
      const uint32_t lb = lane_base<COMPACT>(g, lane);
      float* dst = out + static_cast<long long>(row) * (32LL * KW) + 32 * wcol;
      if constexpr (Form<Q>::kPair) {
        uint32_t nb[4];
        planes_to_nibbles<Q>(P, nb, bc);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const __half2 w2 = *reinterpret_cast<const __half2*>(g_dsmem + lut_offset<COMPACT>(nb[r], lb, j));
            dst[8 * j + r] = __low2float(w2);        // low nibble: column 8j + r
            dst[8 * j + 4 + r] = __high2float(w2);   // high nibble: column 8j + 4 + r
          }
      } else {
        uint32_t b8[8];
        planes_to_bytes<Q>(P, b8, bc);
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int b = 0; b < 4; ++b)
            dst[8 * b + r] = *reinterpret_cast<const float*>(g_dsmem + lut_offset<COMPACT>(b8[r], lb, b));
      }
    }
  }
}

template <int Q>
__global__ void __launch_bounds__(kThreads, 1) dequant_check_kernel(const uint32_t* planes,
                                                                     const uint16_t* lut, int N,
                                                                     int KW, float* out,
                                                                     const BitConsts bc,
                                                                     int32_t* status) {
  constexpr bool C = compact_q<Q>();
  for (int n0 = blockIdx.x * 64; n0 < N; n0 += gridDim.x * 64) {
    const int rows = min(64, N - n0);   // 64, or 32 on a ragged last pass
    if (C || rows == 32) {
      for (int grp = 0; grp < rows / 32; ++grp)
        dequant_check_pass<Q, 1, C>(planes, lut, N, KW, n0 + 32 * grp, out, bc, status);
    } else if constexpr (!C) {
      dequant_check_pass<Q, 2, false>(planes, lut, N, KW, n0, out, bc, status);
    }
  }
}

}  // namespace

cudaError_t launch_index_check(const uint32_t* planes, int N, int K, int q, bool nibbles,
                               uint8_t* idx, cudaStream_t s) {
  const BitConsts bc = make_bit_consts();
  const long long total = static_cast<long long>(N) * (K / 32);
  const int grid = static_cast<int>(std::min<long long>((total + 255) / 256, 64LL * sm_count()));
  const int KW = K / 32;
#define PW_IDX(QQ, NB) index_check_kernel<QQ, NB><<<grid, 256, 0, s>>>(planes, N, KW, idx, bc)
  if (nibbles) {
    switch (q) {
      case 3: PW_IDX(3, true); break;
      case 4: PW_IDX(4, true); break;
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (q) {
      case 3: PW_IDX(3, false); break;
      case 4: PW_IDX(4, false); break;
      case 5: PW_IDX(5, false); break;
      case 6: PW_IDX(6, false); break;
      case 8: PW_IDX(8, false); break;
      default: return cudaErrorInvalidValue;
    }
  }
#undef PW_IDX
  return cudaGetLastError();
}

cudaError_t launch_dequant_check(const uint32_t* planes, const uint16_t* lut, int N, int K, int q,
                                 float* out, int32_t* status, cudaStream_t s) {
  cudaError_t e = setup_once(kSetupDecode, configure_decode);
  if (e != cudaSuccess) return e;
  const BitConsts bc = make_bit_consts();
  const int KW = K / 32;
  const int grid = std::min((N + 63) / 64, 2 * sm_count());
#define PW_DQ(QQ)                                                                              \
  do {                                                                                         \
    e = cudaFuncSetAttribute(dequant_check_kernel<QQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             static_cast<int>(kSmemBytes));                                    \
    if (e != cudaSuccess) return e;                                                            \
    dequant_check_kernel<QQ><<<grid, kThreads, kSmemBytes, s>>>(planes, lut, N, KW, out, bc, status); \
  } while (0)
  switch (q) {
    case 3: PW_DQ(3); break;
    case 4: PW_DQ(4); break;
    case 5: PW_DQ(5); break;
    case 6: PW_DQ(6); break;
    case 8: PW_DQ(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef PW_DQ
  return cudaGetLastError();
}

int decode_max_pairs() { return kMaxPairs; }
int decode_max_experts() { return kMaxExperts; }

// The decode trace of the last gate_up launch (zeros where nothing was
// recorded); returns false when tracing is compiled out.
bool decode_trace_read(void* host, size_t bytes, cudaError_t* err) {
#ifdef PW_TRACE
  *err = cudaMemcpyFromSymbol(host, g_dtrace,
                              sizeof(DecodeTrace) < bytes ? sizeof(DecodeTrace) : bytes);
  return true;
#else
  (void)host;
  (void)bytes;
  *err = cudaSuccess;
  return false;
#endif
}

size_t decode_trace_bytes() { return sizeof(DecodeTrace); }

namespace {

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Clears the decode trace before a gate_up launch (nothing without PW_TRACE).
cudaError_t decode_trace_clear(cudaStream_t stream) {
#ifdef PW_TRACE
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_dtrace);
  if (e != cudaSuccess) return e;
  return cudaMemsetAsync(p, 0, sizeof(DecodeTrace), stream);
#else
  (void)stream;
  return cudaSuccess;
#endif
}

// Routed slots of a call: one per (expert, group of up to kTG pairs), so at
// most the pairs, and at most E + P / kTG.
size_t max_slots(const pw_moe_shape& s) {
  const size_t P = static_cast<size_t>(s.T) * s.k;
  const size_t by_groups = static_cast<size_t>(s.E) + P / kTG;
  return P < by_groups ? P : by_groups;
}

// Down blocks with at least this many word columns (K = I >= 8192) may split
// each row range's K over two tiles (calls whose down tiles fill fewer than
// two rounds of the grid), the second half's partial sums in y2.
constexpr int kSplitDownMinKW = 256;

struct WsSizes {
  size_t xs, xp, hs, hp, y, offsets, perm, routed, ctl, arrive, gu_done, y2;
};

WsSizes ws_sizes(const pw_moe_shape& s) {
  const size_t P = static_cast<size_t>(s.T) * s.k;
  WsSizes z;
  z.xs = round256(4 * static_cast<size_t>(s.T) * s.H);
  z.xp = round256(kRecBytes * static_cast<size_t>(s.T) * (s.H / 32));
  z.hs = round256(4 * P * s.I);
  z.hp = round256(kRecBytes * P * (s.I / 32));
  z.y = round256(4 * P * s.H);
  z.offsets = round256(4 * (static_cast<size_t>(s.E) + 1));
  z.perm = round256(4 * P);
  z.routed = round256(sizeof(SlotInfo) * max_slots(s));
  z.ctl = 256;
  z.arrive = round256(4 * static_cast<size_t>(s.H / 32));
  z.gu_done = round256(4 * P);
  z.y2 = (s.I / 32 >= kSplitDownMinKW) ? round256(4 * P * s.H) : 0;
  return z;
}

// A launch that may start while the previous kernel on the stream finishes
// (programmatic dependent launch); the kernel waits for it with
// griddepcontrol.wait before it depends on its results.
template <typename Kernel, typename... Args>
cudaError_t launch_dependent(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The call is large enough for the GEMM launches to pay off and the GEMM
// kernels support the shape.
bool hybrid_possible(const pw_moe_shape& s) {
  return s.T >= kHybridMinTokens && prefill_shape_ok(s);
}

}  // namespace

// Byte ranges of a decode workspace a caller may read back (test hooks):
// 0 offsets, 1 perm, 2 hidden states in fp32 form, 3 in fp16 records.
int decode_ws_section(const pw_moe_shape& shape, int section, size_t* offset, size_t* bytes) {
  const WsSizes z = ws_sizes(shape);
  const size_t starts[5] = {0, z.xs, z.xs + z.xp, z.xs + z.xp + z.hs, z.xs + z.xp + z.hs + z.hp};
  const size_t off_offsets = starts[4] + z.y;
  switch (section) {
    case 0: *offset = off_offsets; *bytes = 4 * (static_cast<size_t>(shape.E) + 1); return 0;
    case 1: *offset = off_offsets + z.offsets; *bytes = 4 * static_cast<size_t>(shape.T) * shape.k; return 0;
    case 2: *offset = 0; *bytes = 4 * static_cast<size_t>(shape.T) * shape.H; return 0;
    case 3: *offset = z.xs; *bytes = kRecBytes * static_cast<size_t>(shape.T) * (shape.H / 32); return 0;
    default: return -1;
  }
}

// Workspace: hidden states [T][H] fp32 form | the same as fp16 records
// [T][H/32] | h [T*k][I] fp32 form | h as fp16 records [T*k][I/32] | y
// [T*k][H] fp32 | offsets [E+1] | perm [T*k] | routed lists [E] x 2 | control
// words | arrival counters [H/32] | gate_up tiles done [E] | (in calls of at
// least kHybridMinTokens tokens) the GEMM kernels' scratch.
size_t decode_workspace_bytes(const pw_moe_shape& s, bool hybrid) {
  const WsSizes z = ws_sizes(s);
  const size_t base = z.xs + z.xp + z.hs + z.hp + z.y + z.offsets + z.perm + 2 * z.routed + z.ctl +
                      z.arrive + z.gu_done + z.y2;
  return base + ((hybrid && hybrid_possible(s)) ? heavy_scratch_bytes(s) : 0);
}

cudaError_t launch_decode(const LayerArgs& a, void* ws, cudaStream_t stream, bool hybrid) {
  cudaError_t e0 = setup_once(kSetupDecode, configure_decode);
  if (e0 != cudaSuccess) return e0;
  const int sms = sm_count();
  const int n_pairs = a.T * a.k;
  if (n_pairs == 0) return cudaSuccess;
  pw_moe_shape shape{a.T, a.H, a.I, a.E, a.k};
  const WsSizes z = ws_sizes(shape);
  char* p = static_cast<char*>(ws);
  DecodeWs w;
  w.xs = reinterpret_cast<float*>(p); p += z.xs;
  w.xp = p; p += z.xp;
  w.hs = reinterpret_cast<float*>(p); p += z.hs;
  w.hp = p; p += z.hp;
  w.y = reinterpret_cast<float*>(p); p += z.y;
  w.offsets = reinterpret_cast<int*>(p); p += z.offsets;
  w.perm = reinterpret_cast<int*>(p); p += z.perm;
  w.routed_gu = reinterpret_cast<SlotInfo*>(p); p += z.routed;
  w.routed_dn = reinterpret_cast<SlotInfo*>(p); p += z.routed;
  w.ctl = reinterpret_cast<int*>(p); p += z.ctl;
  w.arrive = reinterpret_cast<int*>(p); p += z.arrive;
  w.gu_done = reinterpret_cast<int*>(p); p += z.gu_done;
  w.y2 = z.y2 ? reinterpret_cast<float*>(p) : nullptr; p += z.y2;
  const bool heavy = hybrid && hybrid_possible(shape);
  w.heavy_min = heavy ? kHeavyMinTokens : 0;
  // grids: at most one tile per resident CTA (2 per SM)
  const int slots = static_cast<int>(max_slots(shape));
  const int resident = 2 * sms;
  const int gu_tiles = slots * (a.I / kPairsPerTile);
  // long down blocks in calls with few down tiles split each range's K in two
  // (not with the GEMM kernels, whose rows of y have no second half)
  w.dn_ks = (!heavy && z.y2 && slots * ((a.H + kDownRows - 1) / kDownRows) < 2 * resident) ? 2 : 1;
  const int dn_tiles = slots * ((a.H + kDownRows - 1) / kDownRows) * w.dn_ks;

  const size_t prep_smem = sizeof(int) * static_cast<size_t>(a.E) * (3 + kPrepWarps);
  if (prep_smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_prep_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(prep_smem));
    if (e != cudaSuccess) return e;
  }
  const long long n4 = static_cast<long long>(a.T) * a.H / 4;
  const long long conv = (n4 + kPrepThreads - 1) / kPrepThreads;
  const int prep_grid = 1 + static_cast<int>(conv < 4 * sms ? conv : 4 * sms);
  // Small calls (the down grid leaves SM slots free) launch the prep early
  // and let the down grid release it: it becomes resident while the previous
  // call's down grid runs and starts the moment that grid completes.
  // Larger calls gain nothing from it (every slot is busy) and launch it
  // plainly.  Either way the prep waits for the previous kernel first.
  w.early_next = dn_tiles < resident ? 1 : 0;
  cudaError_t e;
  if (w.early_next) {
    e = launch_dependent(decode_prep_kernel, dim3(prep_grid), dim3(kPrepThreads), prep_smem,
                         stream, a, w);
  } else {
    decode_prep_kernel<<<prep_grid, kPrepThreads, prep_smem, stream>>>(a, w);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  if (heavy) {
    e = launch_heavy(a, w.offsets, w.perm, w.y, p, kHeavyMinTokens, stream);
    if (e != cudaSuccess) return e;
  }

  const BitConsts bc = make_bit_consts();
  if ((e = decode_trace_clear(stream)) != cudaSuccess) return e;
  if ((e = record_timing(g_timing.before, stream)) != cudaSuccess) return e;
  e = launch_dependent(decode_gateup_kernel, dim3(gu_tiles < resident ? gu_tiles : resident),
                       dim3(kThreads), kSmemBytes, stream, a, w, bc);
  if (e != cudaSuccess) return e;
  if ((e = record_timing(g_timing.after, stream)) != cudaSuccess) return e;
  const dim3 dn_grid(dn_tiles < resident ? dn_tiles : resident);
  if (w.dn_ks == 2)
    return launch_dependent(decode_down_kernel<2>, dn_grid, dim3(kThreads), kSmemBytes, stream,
                            a, w, bc);
  return launch_dependent(decode_down_kernel<1>, dn_grid, dim3(kThreads), kSmemBytes, stream, a,
                          w, bc);
}

}  // namespace pw
