// Fused mixed-precision MoE layer, prefill path (many tokens per expert).
//
// PagedWeight, "Core components" 3 (fused mixed-precision kernel): every
// block is read from its top q_i bitplanes and LUT at its own bitwidth.  With
// hundreds of tokens per expert the layer is a dense contraction, so this path
// dequantises weight tiles into shared memory and runs them through the
// tensor cores:
//
//   permute    pairs grouped by expert (offsets, perm)          [pw_route.cu]
//   gather     xg[pos] = fp16(hidden[perm[pos] / k])            (one pass)
//   gate_up    per (expert, 64 gate/up row pairs, 512 tokens):  D = W_gu x^T
//              in TMEM, epilogue h = SiLU(g) * u -> fp16 h[pos]
//   down       per (expert, 128 down rows, 512 tokens):         D = W_dn h^T,
//              epilogue y[pair] (fp32)
//   combine    out[t] = sum_j w_tj * y[t*k + j], j order        (one pass)
//
// GEMM kernel (one CTA per SM, persistent over a static tile list; 14 warps):
//   warps 0-7   dequant producers in two sets of four that take alternate
//               k-steps; thread r of a set owns A-tile row r.  Per k-step (32
//               columns) it loads one word of each of the row's top q planes
//               (a word column of consecutive rows is contiguous), rebuilds
//               the 32 indices with a byte transpose and an 8x8 bit-matrix
//               transpose, looks them up in the row's LUT (fp16, shared
//               memory; a byte permute forms each address) and writes the
//               fp16 row into the 64-byte-swizzled, K-major A stage.
//   warps 8-11  epilogue: drain the TMEM accumulator (lane quarter = warp%4).
//   warp 12     TMA producer for the token operand (fp16 rows, 64B swizzle).
//   warp 13     allocates all 512 TMEM columns; lane 0 issues per k-step two
//               K=16 steps of two tcgen05.mma (M=128, N=256 each, fp16 x
//               fp16 -> fp32) into columns [0,256) and [256,512).
// A weight tile is dequantised once per 512 tokens.  Stages are handed over
// with mbarriers; every wait is bounded and a timeout latches PW_ERR_TIMEOUT
// and unwinds without trapping.
//
// Operand precision: the weights are exact fp16 LUT values; hidden states are
// converted bf16 -> fp16 (exact for |x| in fp16's normal range, |x| < 65504);
// h is stored as fp16; all accumulation is fp32.
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
constexpr int NST = 3;                  // pipeline stages
constexpr int kDqThreads = 256;         // warps 0-7
constexpr int kEpiWarp0 = 8;            // warps 8-11
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr uint32_t kAStage = BM * BK * 2;     // 8 KB
constexpr uint32_t kBHalf = BNH * BK * 2;     // 16 KB per 256 tokens
constexpr uint32_t kBStage = 2 * kBHalf;      // 32 KB
constexpr uint32_t kLutBytes = 256 * BM * 2;  // fp16 [256][128]
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSpinLimit = 1u << 24;
constexpr int kMaxExperts = 1024;

// Shared memory (offsets from the dynamic base, which must be 1024-aligned):
// the LUT sits at offset 0 so that lookups address the dynamic symbol with a
// register offset only.
constexpr uint32_t kOffLut = 0;
constexpr uint32_t kOffA = kOffLut + kLutBytes;
constexpr uint32_t kOffB = kOffA + NST * kAStage;
constexpr uint32_t kOffBar = kOffB + NST * kBStage;            // 8-byte barriers
constexpr int kBarFullA = 0, kBarFullB = NST, kBarEmpty = 2 * NST, kBarAccFull = 3 * NST,
              kBarAccEmpty = 3 * NST + 1, kBarFinal = 3 * NST + 2, kNumBars = 3 * NST + 3;
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;          // tmem base, abort flag
constexpr uint32_t kOffPrefix = kOffMisc + 16;                 // tile prefix [E+1]
constexpr size_t kSmemBytes = kOffPrefix + 4 * (kMaxExperts + 1);

extern __shared__ __align__(1024) unsigned char g_psmem[];

enum Mode { kGateUp = 0, kDown = 1 };

struct GemmArgs {
  int32_t H, I, E, k, n_pairs;
  const pw_block_entry* table;
  const int32_t* offsets;   // [E+1]
  const int32_t* perm;      // [n_pairs]
  __half* h_ws;             // [n_pairs][I] (gate_up writes, down reads through TMA)
  float* y_ws;              // [n_pairs][H]
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
                                          int32_t* status) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  latch_status(status, PW_ERR_TIMEOUT);
  return false;
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

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc)
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

// ---------------------------------------------------------------- tile list

struct Tile {
  int e, m, n;  // expert, row tile, token tile
};

__device__ __forceinline__ int m_tiles(Mode mode, const GemmArgs& a) {
  return mode == kGateUp ? a.I / 64 : a.H / BM;
}

// Tile t of the list ordered (expert, row tile, token tile), token tile fastest.
__device__ __forceinline__ Tile tile_at(int t, const int* prefix, int E, const int32_t* offsets) {
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
  r.m = local / nt;
  r.n = local % nt;
  return r;
}

// Row of the block behind A-tile row r.  gate_up tiles interleave gate and up
// rows (even r: gate row, odd r: the matching up row) so that the epilogue
// pairs them with one lane exchange.
__device__ __forceinline__ int block_row(Mode mode, const GemmArgs& a, int m, int r) {
  if (mode == kGateUp) return (r & 1) ? a.I + m * 64 + (r >> 1) : m * 64 + (r >> 1);
  return m * BM + r;
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

// ---------------------------------------------------------------- dequant

// Byte offset of row r's entries inside a LUT line: rows r and r+64 share
// one 4-byte word, so the 32 consecutive rows of a warp use 32 different
// banks.  Fits in one byte (at most 254).
__device__ __forceinline__ uint32_t lut_row_bytes(int r) {
  return (static_cast<uint32_t>(r & 63) << 2) | (static_cast<uint32_t>(r >> 6) << 1);
}

// LUT of the tile's rows: byte v*256 + lut_row_bytes(r) holds LUT_q[row(r)][v]
// (fp16).  The 256 dequant threads split each row's entries in two halves.
template <int Q>
__device__ __forceinline__ void load_lut(const uint16_t* lut, int grow, int r, int half) {
  constexpr int kEnt = 1 << Q;
  constexpr int kVec = kEnt / 8;
  const uint4* src = reinterpret_cast<const uint4*>(lut + static_cast<long long>(grow) * kEnt);
#pragma unroll 4
  for (int vec = half; vec < kVec; vec += 2) {
    const uint4 raw = __ldg(src + vec);
    const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint16_t*>(g_psmem + kOffLut + (vec * 8 + j) * 256 + lut_row_bytes(r)) =
          h[j];
  }
}

template <int Q>
__device__ __forceinline__ void load_words(const uint32_t* row_planes, long long plane_stride,
                                           long long N, int ks, uint32_t (&w)[Q]) {
#pragma unroll
  for (int p = 0; p < Q; ++p) w[p] = __ldg(row_planes + p * plane_stride + ks * N);
}

// Thread r: fill A-stage row r with the 32 weights whose plane words are w.
template <int Q>
__device__ __forceinline__ void dequant_kstep(const uint32_t (&w)[Q], int r, uint32_t a_stage,
                                              const BitConsts& bc) {
  uint32_t ib[8];
  planes_to_index_bytes<Q>(w, ib, bc);
  const uint32_t rb = lut_row_bytes(r);
  const uint32_t row_base = a_stage + r * 64;
  const uint32_t sw = (r >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) {   // 16-byte chunk c = columns 8c .. 8c+7
    uint32_t packed[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t word = ib[2 * c + h];
      uint32_t v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t off = __byte_perm(word, rb, 0x6504 | (j << 4));
        v[j] = *reinterpret_cast<const uint16_t*>(g_psmem + off);
      }
      packed[2 * h] = __byte_perm(v[0], v[1], 0x5410);
      packed[2 * h + 1] = __byte_perm(v[2], v[3], 0x5410);
    }
    const uint32_t dst = row_base + ((c ^ sw) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[0]),
                 "r"(packed[1]), "r"(packed[2]), "r"(packed[3])
                 : "memory");
  }
}

template <int Q>
__device__ void dequant_tile(const GemmArgs& a, Mode mode, const pw_block_entry& ent, int m,
                             int ksteps, uint32_t it_base, int set, int r, uint32_t bar_base,
                             volatile int* abort, const BitConsts& bc) {
  const int grow = block_row(mode, a, m, r);
  named_sync_dq();                      // both sets are done with the previous tile's LUT
  if (!*abort) load_lut<Q>(ent.lut, grow, r, set);
  named_sync_dq();
  const long long N = (mode == kGateUp) ? 2LL * a.I : a.H;
  const long long KW = ((mode == kGateUp) ? a.H : a.I) / 32;
  const long long plane_stride = N * KW;
  const uint32_t* row_planes = ent.planes + grow;
  const uint32_t a_base = smem_u32(g_psmem) + kOffA;
  // plane words are loaded two k-steps (of this set) ahead
  uint32_t n1[Q], n2[Q];
  if (set < ksteps) load_words<Q>(row_planes, plane_stride, N, set, n1);
  if (set + 2 < ksteps) load_words<Q>(row_planes, plane_stride, N, set + 2, n2);
  for (int ks = set; ks < ksteps; ks += 2) {
    uint32_t cur[Q];
#pragma unroll
    for (int p = 0; p < Q; ++p) {
      cur[p] = n1[p];
      n1[p] = n2[p];
    }
    if (ks + 4 < ksteps) load_words<Q>(row_planes, plane_stride, N, ks + 4, n2);
    const uint32_t it = it_base + ks;
    const int stage = it % NST;
    const uint32_t par = (it / NST) & 1u;
    if (*abort) continue;
    if (!mbar_wait(bar_base + 8 * (kBarEmpty + stage), par ^ 1u, abort, a.status)) continue;
    dequant_kstep<Q>(cur, r, a_base + stage * kAStage, bc);
    fence_proxy_async();
    mbar_arrive(bar_base + 8 * (kBarFullA + stage));
  }
}

// ---------------------------------------------------------------- epilogue

__device__ void epilogue(const GemmArgs& a, Mode mode, const Tile& tile, int pos0, int ntok,
                         bool usable, uint32_t tmem_base, int quarter, int lane, uint32_t bar_base,
                         uint32_t acc_par, volatile int* abort) {
  const int r = quarter * 32 + lane;
  if (usable) {
    if (*abort || !mbar_wait(bar_base + 8 * kBarAccFull, acc_par, abort, a.status)) return;
    tc_fence_after();
  }
  for (int c = 0; c < BN / 32; ++c) {
    if (c * 32 >= ntok) break;
    float v[32];
    if (usable) {
      tmem_ld32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + c * 32, v);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    }
    if (mode == kGateUp) {
      if (!usable) continue;  // h of a skipped expert is never read
      const int col = tile.m * 64 + (r >> 1);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
        const int n = c * 32 + j;
        if ((lane & 1) == 0 && n < ntok) {
          const float g = v[j], u = other;
          const float h = g / (1.f + expf(-g)) * u;
          a.h_ws[static_cast<long long>(pos0 + n) * a.I + col] = __float2half_rn(h);
        }
      }
    } else {
      const int row = tile.m * BM + r;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int n = c * 32 + j;
        if (n < ntok) {
          const int pair = a.perm[pos0 + n];
          a.y_ws[static_cast<long long>(pair) * a.H + row] = v[j];
        }
      }
    }
  }
  if (usable) {
    tc_fence_before();
    mbar_arrive(bar_base + 8 * kBarAccEmpty);
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
  int* prefix = reinterpret_cast<int*>(g_psmem + kOffPrefix);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = m_tiles(mode, a);
  const int K = (mode == kGateUp) ? a.H : a.I;
  const int ksteps = K / BK;
  if (sbase & 1023u) {   // the swizzled stages need a 1024-byte aligned base
    if (tid == 0) latch_status(a.status, PW_ERR_CUDA);
    return;
  }

  if (tid == 0) {
    *abort = 0;
    int run = 0;
    for (int e = 0; e < a.E; ++e) {
      prefix[e] = run;
      run += mt * ((a.offsets[e + 1] - a.offsets[e] + BN - 1) / BN);
    }
    prefix[a.E] = run;
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar_base + 8 * (kBarFullA + i), kDqThreads / 2);
      mbar_init(bar_base + 8 * (kBarFullB + i), 1);
      mbar_init(bar_base + 8 * (kBarEmpty + i), 1);
    }
    mbar_init(bar_base + 8 * kBarAccFull, 1);
    mbar_init(bar_base + 8 * kBarAccEmpty, 128);
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

  if (warp < 8) {
    // ---- dequant producers: set 0 = warps 0-3 (even k-steps), set 1 = warps 4-7
    const int set = warp >> 2, r = tid & 127;
    uint32_t it_base = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tile = tile_at(t, prefix, a.E, a.offsets);
      const bool usable = tile_usable(mode, a, tile.e);
      if (!usable) continue;
      const pw_block_entry ent = a.table[2 * tile.e + (mode == kGateUp ? 0 : 1)];
      switch (ent.q) {
        case 3: dequant_tile<3>(a, mode, ent, tile.m, ksteps, it_base, set, r, bar_base, abort, bc); break;
        case 4: dequant_tile<4>(a, mode, ent, tile.m, ksteps, it_base, set, r, bar_base, abort, bc); break;
        case 5: dequant_tile<5>(a, mode, ent, tile.m, ksteps, it_base, set, r, bar_base, abort, bc); break;
        case 6: dequant_tile<6>(a, mode, ent, tile.m, ksteps, it_base, set, r, bar_base, abort, bc); break;
        default: dequant_tile<8>(a, mode, ent, tile.m, ksteps, it_base, set, r, bar_base, abort, bc); break;
      }
      it_base += ksteps;
    }
  } else if (warp < kTmaWarp) {
    // ---- epilogue
    const int quarter = warp - kEpiWarp0;
    uint32_t acc_it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tile = tile_at(t, prefix, a.E, a.offsets);
      const int pos0 = a.offsets[tile.e] + tile.n * BN;
      const int ntok = min(BN, a.offsets[tile.e + 1] - pos0);
      const bool usable = tile_usable(mode, a, tile.e);
      if (!usable && quarter == 0 && lane == 0) report_unusable(mode, a, tile.e);
      epilogue(a, mode, tile, pos0, ntok, usable, tmem_base, quarter, lane, bar_base, acc_it & 1u,
               abort);
      if (usable) ++acc_it;
    }
  } else if (warp == kTmaWarp) {
    // ---- TMA producer for the token operand
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
      uint32_t it = 0;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        const Tile tile = tile_at(t, prefix, a.E, a.offsets);
        if (!tile_usable(mode, a, tile.e)) continue;
        const int pos0 = a.offsets[tile.e] + tile.n * BN;
        const int ntok = min(BN, a.offsets[tile.e + 1] - pos0);
        const int halves = ntok > BNH ? 2 : 1;
        for (int s = 0; s < ksteps; ++s, ++it) {
          const int stage = it % NST;
          const uint32_t par = (it / NST) & 1u;
          if (!mbar_wait(bar_base + 8 * (kBarEmpty + stage), par ^ 1u, abort, a.status)) break;
          const uint32_t full = bar_base + 8 * (kBarFullB + stage);
          mbar_arrive_tx(full, halves * kBHalf);
          for (int h = 0; h < halves; ++h)
            tma_load_2d(sbase + kOffB + stage * kBStage + h * kBHalf, &tmap_b, s * BK,
                        pos0 + h * BNH, full);
        }
      }
      if (*abort) {
        // let the copies this thread issued land before the CTA unwinds
        for (uint32_t j = (it > NST ? it - NST : 0); j < it; ++j) {
          const uint32_t bar = bar_base + 8 * (kBarFullB + j % NST);
          for (uint32_t i = 0; i < kSpinLimit && !mbar_try(bar, (j / NST) & 1u); ++i) {
          }
        }
      }
    }
  } else {
    // ---- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool issued = false;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        const Tile tile = tile_at(t, prefix, a.E, a.offsets);
        if (!tile_usable(mode, a, tile.e)) continue;
        const int pos0 = a.offsets[tile.e] + tile.n * BN;
        const int ntok = min(BN, a.offsets[tile.e + 1] - pos0);
        const int n0 = min(BNH, (ntok + 15) & ~15);
        const int n1 = ntok > BNH ? ((ntok - BNH + 15) & ~15) : 0;
        const uint32_t id0 = make_idesc(n0), id1 = make_idesc(n1 > 0 ? n1 : 16);
        if (!mbar_wait(bar_base + 8 * kBarAccEmpty, (acc_it & 1u) ^ 1u, abort, a.status)) break;
        tc_fence_after();
        for (int s = 0; s < ksteps; ++s, ++it) {
          const int stage = it % NST;
          const uint32_t par = (it / NST) & 1u;
          if (!mbar_wait(bar_base + 8 * (kBarFullA + stage), par, abort, a.status)) break;
          if (!mbar_wait(bar_base + 8 * (kBarFullB + stage), par, abort, a.status)) break;
          tc_fence_after();
          const uint32_t a_addr = sbase + kOffA + stage * kAStage;
          const uint32_t b_addr = sbase + kOffB + stage * kBStage;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
            mma_f16(tmem_base, smem_desc(a_addr + kk * 32), smem_desc(b_addr + kk * 32), id0, acc);
            if (n1 > 0)
              mma_f16(tmem_base + BNH, smem_desc(a_addr + kk * 32),
                      smem_desc(b_addr + kBHalf + kk * 32), id1, acc);
          }
          issued = true;
          mma_commit(bar_base + 8 * (kBarEmpty + stage));
        }
        if (*abort) break;
        mma_commit(bar_base + 8 * kBarAccFull);
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

// xg[pos][c] = fp16(hidden[perm[pos] / k][c]); positions past the routed
// pairs are zero.  8 columns per thread.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ hidden,
                                                     const int32_t* __restrict__ perm,
                                                     const int32_t* __restrict__ offsets, int E,
                                                     int k, int H, int n_pairs,
                                                     __half* __restrict__ xg) {
  const long long per_row = H / 8;
  const long long total = static_cast<long long>(n_pairs) * per_row;
  const int valid = offsets[E];
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i / per_row);
    const int c = static_cast<int>(i % per_row) * 8;
    uint4 outv = make_uint4(0, 0, 0, 0);
    if (pos < valid) {
      const int t = perm[pos] / k;
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(hidden + static_cast<long long>(t) * H + c));
      const uint16_t* b = reinterpret_cast<const uint16_t*>(&raw);
      __half2 h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        h[j] = __floats2half2_rn(bf16_bits_to_float(b[2 * j]), bf16_bits_to_float(b[2 * j + 1]));
      outv = *reinterpret_cast<const uint4*>(h);
    }
    *reinterpret_cast<uint4*>(xg + static_cast<long long>(pos) * H + c) = outv;
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y_ws,
                                                      const int32_t* __restrict__ ids,
                                                      const float* __restrict__ wts, int T, int k,
                                                      int E, int H, float* __restrict__ out) {
  const long long total = static_cast<long long>(T) * H;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H);
    const int n = static_cast<int>(i % H);
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int p = t * k + j;
      const int e = ids[p];
      if (e < 0 || e >= E) continue;
      acc = fmaf(wts[p], y_ws[static_cast<long long>(p) * H + n], acc);
    }
    out[i] = acc;
  }
}

// ---------------------------------------------------------------- host side

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  int32_t* offsets;
  int32_t* perm;
  __half* xg;
  __half* h;
  float* y;
};

WsLayout carve_ws(void* ws, const pw_moe_shape& s) {
  const size_t P = static_cast<size_t>(s.T) * s.k;
  char* p = static_cast<char*>(ws);
  WsLayout w;
  w.offsets = reinterpret_cast<int32_t*>(p);
  p += round256(sizeof(int32_t) * (s.E + 1));
  w.perm = reinterpret_cast<int32_t*>(p);
  p += round256(sizeof(int32_t) * P);
  w.xg = reinterpret_cast<__half*>(p);
  p += round256(2 * P * s.H);
  w.h = reinterpret_cast<__half*>(p);
  p += round256(2 * P * s.I);
  w.y = reinterpret_cast<float*>(p);
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

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace

size_t prefill_workspace_bytes(const pw_moe_shape& s) {
  const size_t P = static_cast<size_t>(s.T) * s.k;
  return round256(sizeof(int32_t) * (s.E + 1)) + round256(sizeof(int32_t) * P) +
         round256(2 * P * s.H) + round256(2 * P * s.I) + round256(4 * P * s.H);
}

bool prefill_shape_ok(const pw_moe_shape& s) {
  return s.H % BM == 0 && s.I % 64 == 0 && s.E <= kMaxExperts;
}

int prefill_min_pairs(const pw_moe_shape& s) { return prefill_shape_ok(s) ? 1024 : INT_MAX; }

cudaError_t launch_prefill(const LayerArgs& la, void* ws, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(dq_gemm_kernel<kGateUp>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dq_gemm_kernel<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  pw_moe_shape s{la.T, la.H, la.I, la.E, la.k};
  const int n_pairs = la.T * la.k;
  if (n_pairs == 0) return cudaSuccess;
  WsLayout w = carve_ws(ws, s);
  cudaError_t e = launch_permute(la.topk_ids, n_pairs, la.E, w.offsets, w.perm, nullptr, la.status,
                                 stream);
  if (e != cudaSuccess) return e;
  const long long gwork = static_cast<long long>(n_pairs) * (la.H / 8);
  const int gblocks = static_cast<int>(std::min<long long>((gwork + 255) / 256, 152LL * 32));
  gather_kernel<<<gblocks, 256, 0, stream>>>(la.hidden, w.perm, w.offsets, la.E, la.k, la.H,
                                             n_pairs, w.xg);
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
  g.h_ws = w.h;
  g.y_ws = w.y;
  g.status = la.status;
  const int grid = num_sms();
  const BitConsts bc = make_bit_consts();
  dq_gemm_kernel<kGateUp><<<grid, kThreads, kSmemBytes, stream>>>(g, map_x, bc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dq_gemm_kernel<kDown><<<grid, kThreads, kSmemBytes, stream>>>(g, map_h, bc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long cwork = static_cast<long long>(la.T) * la.H;
  const int cblocks = static_cast<int>(std::min<long long>((cwork + 255) / 256, 152LL * 32));
  combine_kernel<<<cblocks, 256, 0, stream>>>(w.y, la.topk_ids, la.topk_weights, la.T, la.k, la.E,
                                              la.H, la.out);
  return cudaGetLastError();
}

}  // namespace pw
