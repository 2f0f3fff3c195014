// Fused mixed-precision MoE layer, decode path (few tokens per expert).
//
// PagedWeight, "Core components" 3 (fused mixed-precision kernel): the kernel
// reads every linear block's bitplanes and LUT directly, each block at its own
// committed bitwidth q_i, inside one fused operation.  Two launches:
//
//   gateup: per (routed expert e, tile of 32 gate/up row pairs): read the top
//           q planes of gate rows i and up rows I+i, rebuild the q-bit codes,
//           look them up in each row's LUT, dot with the expert's gathered
//           hidden rows (fp32), then h = SiLU(g) * u -> workspace.
//   down:   per (routed expert e, tile of 64 down rows): same bitplane/LUT
//           read at the down block's q, dot with h -> y for each of e's pairs
//           (workspace).  The last CTA to finish a row tile (a per-tile
//           arrival counter) combines out[t] = sum_j w_tj * y[t*k + j] over
//           the tile in j order, so the output is deterministic.
//
// Work inside a CTA: lane L owns rows (row0 + L) and (row0' + L) of the tile;
// the 8 warps split the K columns and their partial sums meet in shared
// memory.  Per 32 columns a lane loads one word of each of the top q planes
// per row (a word column of consecutive rows is contiguous, so a warp's load
// is one 128-byte line), turns the q words into 32 index bytes with a byte
// transpose and an 8x8 bit-matrix transpose, and looks each index up in its
// row's LUT, which sits in a lane-private shared-memory column: one byte
// permute forms the address (index * 256 + slot * 128 + lane * 4), and every
// lookup of lane L hits bank L.
//
// Each CTA finds its expert itself from topk_ids (count, pick the slot-th
// routed expert, list its pairs in ascending pair order), so no separate
// routing launch is needed on this path.
#include <cuda_fp16.h>

#include "pw_internal.cuh"

namespace pw {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPairsPerTile = 32;   // gate_up tile: 32 gate rows + their 32 up rows
constexpr int kDownRows = 64;       // down tile: two 32-row groups
constexpr int kTG = 4;              // tokens per pass over the weights
constexpr int kCW = 4;              // words per staged activation chunk
constexpr int kCC = kCW * 32;       // columns per staged activation chunk
constexpr int kMaxPairs = 4096;     // T*k limit of this path
constexpr int kMaxExperts = 1024;

// Shared memory (bytes).  The LUT region comes first: entry v of row slot g
// for lane L sits at byte v*256 + g*128 + L*4 (fp32), so a lane's lookups
// always hit bank L and one byte permute turns an 8-bit index into the offset.
constexpr int kLutBytes = 256 * 256;
constexpr int kActBytes = kWarps * kTG * kCC * 4;
constexpr int kRedBytes = kWarps * kTG * 2 * 32 * 4;
constexpr int kCountBytes = kMaxExperts * 4;
constexpr int kPairBytes = kMaxPairs * 4;
constexpr int kOffAct = kLutBytes;
constexpr int kOffRed = kOffAct + kActBytes;
constexpr int kOffCount = kOffRed + kRedBytes;
constexpr int kOffPairs = kOffCount + kCountBytes;
constexpr int kOffMisc = kOffPairs + kPairBytes;
constexpr size_t kSmemBytes = kOffMisc + 64;

struct SmemPtrs {
  unsigned char* lut;
  float* act;
  float* red;
  int* count;
  int* pairs;
  int* misc;
};

__device__ __forceinline__ SmemPtrs carve(unsigned char* base) {
  SmemPtrs s;
  s.lut = base;
  s.act = reinterpret_cast<float*>(base + kOffAct);
  s.red = reinterpret_cast<float*>(base + kOffRed);
  s.count = reinterpret_cast<int*>(base + kOffCount);
  s.pairs = reinterpret_cast<int*>(base + kOffPairs);
  s.misc = reinterpret_cast<int*>(base + kOffMisc);
  return s;
}

struct Route {
  int e;    // routed expert of this CTA's slot, -1 if the slot is empty
  int off;  // number of pairs routed to lower expert ids
  int ne;   // number of pairs routed to e
};

// Whole-CTA: count pairs per expert, pick the slot-th routed expert (ascending
// id), list its pairs ascending into s.pairs.
__device__ Route route_slot(const LayerArgs& a, int slot, const SmemPtrs& s, bool report) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_pairs = a.T * a.k;
  for (int e = tid; e < a.E; e += kThreads) s.count[e] = 0;
  __syncthreads();
  for (int p = tid; p < n_pairs; p += kThreads) {
    const int e = a.topk_ids[p];
    if (e >= 0 && e < a.E) {
      atomicAdd(&s.count[e], 1);
    } else if (report) {
      latch_status(a.status, PW_ERR_BAD_EXPERT_ID);
    }
  }
  __syncthreads();
  if (warp == 0) {
    int routed = 0;
    for (int base = 0; base < a.E; base += 32) {
      const int e = base + lane;
      routed += __popc(__ballot_sync(kFull, e < a.E && s.count[e] > 0));
    }
    if (lane == 0) s.misc[3] = routed;
    int seen = 0, off = 0, found = -1;
    for (int base = 0; base < a.E && found < 0; base += 32) {
      const int e = base + lane;
      const int c = (e < a.E) ? s.count[e] : 0;
      const unsigned mask = __ballot_sync(kFull, c > 0);
      const int n = __popc(mask);
      int part;
      if (slot < seen + n) {
        const int want = slot - seen;
        const bool mine = (c > 0) && (__popc(mask & ((1u << lane) - 1u)) == want);
        const int src = __ffs(__ballot_sync(kFull, mine)) - 1;
        found = base + src;
        part = (lane < src) ? c : 0;
      } else {
        part = c;
        seen += n;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
      off += part;
    }
    if (lane == 0) {
      s.misc[0] = found;
      s.misc[1] = off;
      s.misc[2] = (found >= 0) ? s.count[found] : 0;
    }
    if (found >= 0) {
      int run = 0;
      for (int c0 = 0; c0 < n_pairs; c0 += 32) {
        const int p = c0 + lane;
        const bool hit = (p < n_pairs) && (a.topk_ids[p] == found);
        const unsigned m = __ballot_sync(kFull, hit);
        if (hit) s.pairs[run + __popc(m & ((1u << lane) - 1u))] = p;
        run += __popc(m);
      }
    }
  }
  __syncthreads();
  Route r;
  r.e = s.misc[0];
  r.off = s.misc[1];
  r.ne = s.misc[2];
  return r;
}

// LUT rows of the tile into the lane-private layout: row slot g, lane L,
// entry v -> byte v*256 + g*128 + L*4, as fp32.  Each thread moves 8 fp16
// entries (16 bytes); the stores of a warp hit 32 different banks.
template <int Q, int R>
__device__ __forceinline__ void load_luts(const uint16_t* lut, const int (&row0)[R],
                                          const SmemPtrs& s) {
  constexpr int kEnt = 1 << Q;
  constexpr int kVecPerRow = kEnt / 8;
#pragma unroll
  for (int g = 0; g < R; ++g) {
    for (int i = threadIdx.x; i < 32 * kVecPerRow; i += kThreads) {
      const int L = i & 31, vec = i >> 5;
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
          lut + static_cast<long long>(row0[g] + L) * kEnt + vec * 8));
      const __half* h = reinterpret_cast<const __half*>(&raw);
      unsigned char* dst = s.lut + (vec * 8) * 256 + g * 128 + L * 4;
#pragma unroll
      for (int j = 0; j < 8; ++j) *reinterpret_cast<float*>(dst + j * 256) = __half2float(h[j]);
    }
  }
}

// Byte transpose of four 32-bit words: out[b] = {a0.byte b, a1.byte b,
// a2.byte b, a3.byte b}.
__device__ __forceinline__ void byte_transpose4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t (&out)[4]) {
  const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
  const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

// Transpose of the 8x8 bit matrix held in (lo, hi): byte r = matrix row r,
// bit c = column c  ->  byte c = column c, bit r = row r.  Three delta swaps.
__device__ __forceinline__ void bit_transpose8(uint32_t& lo, uint32_t& hi) {
  uint32_t t;
  t = (lo ^ (lo >> 7)) & 0x00AA00AAu; lo ^= t ^ (t << 7);
  t = (hi ^ (hi >> 7)) & 0x00AA00AAu; hi ^= t ^ (t << 7);
  t = (lo ^ (lo >> 14)) & 0x0000CCCCu; lo ^= t ^ (t << 14);
  t = (hi ^ (hi >> 14)) & 0x0000CCCCu; hi ^= t ^ (t << 14);
  t = (lo ^ (hi << 4)) & 0xF0F0F0F0u; lo ^= t; hi ^= t >> 4;
}

// Q plane words of one row (P[0] = most significant plane) covering 32
// columns -> the q-bit index of every column, one per byte: byte j of ib[m]
// is the index of column 4m + j.  Plane p feeds bit (Q-1-p) of the index;
// for Q <= 4 half of the matrix is zero and the compiler folds it away.
template <int Q>
__device__ __forceinline__ void planes_to_index_bytes(const uint32_t (&P)[Q], uint32_t (&ib)[8]) {
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = (i < Q) ? P[Q - 1 - i] : 0u;
  uint32_t A[4], B[4];
  byte_transpose4(r[0], r[1], r[2], r[3], A);
  byte_transpose4(r[4], r[5], r[6], r[7], B);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    uint32_t lo = A[b], hi = B[b];
    bit_transpose8(lo, hi);
    ib[2 * b] = lo;
    ib[2 * b + 1] = hi;
  }
}

__device__ __forceinline__ float lane4(const float4& v, int j) {
  return (j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w;
}

// Partial dot products of this lane's R rows over the warp's words
// [kw_lo, kw_hi), for NT tokens whose activations `load_chunk` stages per
// kCW-word chunk.  Plane words are loaded one word column ahead.
template <int Q, int R, int NT, class Loader>
__device__ __forceinline__ void rows_dot(const uint32_t* planes, long long plane_stride, int N,
                                         const int (&row)[R], int kw_lo, int kw_hi,
                                         const SmemPtrs& s, const Loader& load_chunk,
                                         float (&acc)[R][NT]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* act = s.act + warp * (kTG * kCC);
  uint32_t lb[R];
#pragma unroll
  for (int g = 0; g < R; ++g) lb[g] = (static_cast<uint32_t>(g) << 7) | (lane << 2);
#pragma unroll
  for (int g = 0; g < R; ++g)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[g][t] = 0.f;
  if (kw_lo >= kw_hi) return;
  uint32_t nxt[R][Q];
#pragma unroll
  for (int g = 0; g < R; ++g)
#pragma unroll
    for (int p = 0; p < Q; ++p)
      nxt[g][p] = __ldg(planes + p * plane_stride + static_cast<long long>(kw_lo) * N + row[g]);
  for (int kw0 = kw_lo; kw0 < kw_hi; kw0 += kCW) {
    const int nw = min(kCW, kw_hi - kw0);
    __syncwarp();
    load_chunk(act, kw0 * 32, nw * 32);
    __syncwarp();
    for (int ww = 0; ww < nw; ++ww) {
      uint32_t cur[R][Q];
#pragma unroll
      for (int g = 0; g < R; ++g)
#pragma unroll
        for (int p = 0; p < Q; ++p) cur[g][p] = nxt[g][p];
      const int kn = kw0 + ww + 1;
      if (kn < kw_hi) {
#pragma unroll
        for (int g = 0; g < R; ++g)
#pragma unroll
          for (int p = 0; p < Q; ++p)
            nxt[g][p] = __ldg(planes + p * plane_stride + static_cast<long long>(kn) * N + row[g]);
      }
      uint32_t ib[R][8];
#pragma unroll
      for (int g = 0; g < R; ++g) planes_to_index_bytes<Q>(cur[g], ib[g]);
      const float* xa = act + ww * 32;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float4 xv[NT];
#pragma unroll
        for (int tk = 0; tk < NT; ++tk)
          xv[tk] = *reinterpret_cast<const float4*>(xa + tk * kCC + 4 * m);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int g = 0; g < R; ++g) {
            const uint32_t off = __byte_perm(ib[g][m], lb[g], 0x6504 | (j << 4));
            const float w = *reinterpret_cast<const float*>(s.lut + off);
#pragma unroll
            for (int tk = 0; tk < NT; ++tk) acc[g][tk] = fmaf(lane4(xv[tk], j), w, acc[g][tk]);
          }
        }
      }
    }
  }
}

__device__ __forceinline__ void warp_range(int KW, int& lo, int& hi) {
  const int warp = threadIdx.x >> 5;
  lo = (warp * KW) / kWarps;
  hi = ((warp + 1) * KW) / kWarps;
}

// ---------------------------------------------------------------- gate_up

template <int Q, int NT>
__device__ void gateup_group(const LayerArgs& a, const Route& r, const pw_block_entry& ent,
                             int i0, int g0, int nt, const SmemPtrs& s, float* h_ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KW = a.H / 32;
  const int N = 2 * a.I;
  const long long plane_stride = static_cast<long long>(N) * KW;
  const int row[2] = {i0 + lane, a.I + i0 + lane};
  int lo, hi;
  warp_range(KW, lo, hi);
  int tok[NT];
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) tok[tk] = (tk < nt) ? s.pairs[g0 + tk] / a.k : -1;
  auto loader = [&](float* act, int c0, int cols) {
    const int c = lane * 4;
#pragma unroll
    for (int tk = 0; tk < NT; ++tk) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tok[tk] >= 0 && c < cols) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(
            a.hidden + static_cast<long long>(tok[tk]) * a.H + c0 + c));
        v = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                        __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
      }
      *reinterpret_cast<float4*>(act + tk * kCC + c) = v;
    }
  };
  float acc[2][NT];
  rows_dot<Q, 2, NT>(ent.planes, plane_stride, N, row, lo, hi, s, loader, acc);
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) {
    s.red[((warp * kTG + tk) * 2 + 0) * 32 + lane] = acc[0][tk];
    s.red[((warp * kTG + tk) * 2 + 1) * 32 + lane] = acc[1][tk];
  }
  __syncthreads();
  if (threadIdx.x < 32 * nt) {
    const int tk = threadIdx.x >> 5;
    float g = 0.f, u = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      g += s.red[((w * kTG + tk) * 2 + 0) * 32 + lane];
      u += s.red[((w * kTG + tk) * 2 + 1) * 32 + lane];
    }
    const float h = g / (1.f + expf(-g)) * u;
    h_ws[static_cast<long long>(r.off + g0 + tk) * a.I + i0 + lane] = h;
  }
  __syncthreads();
}

template <int Q>
__device__ void gateup_tile(const LayerArgs& a, const Route& r, const pw_block_entry& ent,
                            int i0, const SmemPtrs& s, float* h_ws) {
  const int row0[2] = {i0, a.I + i0};
  load_luts<Q, 2>(ent.lut, row0, s);
  __syncthreads();
  for (int g0 = 0; g0 < r.ne; g0 += kTG) {
    const int nt = min(kTG, r.ne - g0);
    if (nt == 1) gateup_group<Q, 1>(a, r, ent, i0, g0, nt, s, h_ws);
    else if (nt == 2) gateup_group<Q, 2>(a, r, ent, i0, g0, nt, s, h_ws);
    else gateup_group<Q, 4>(a, r, ent, i0, g0, nt, s, h_ws);
  }
}

__global__ void __launch_bounds__(kThreads, 2) decode_gateup_kernel(const LayerArgs a, float* h_ws,
                                                                    int* tile_count) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const SmemPtrs s = carve(smem_raw);
  // Zero the output (covers calls where no pair has a valid expert) and the
  // down kernel's per-tile arrival counters; the down kernel runs after this
  // grid has completed.
  {
    const long long total = static_cast<long long>(a.T) * a.H;
    const long long cta = blockIdx.y * static_cast<long long>(gridDim.x) + blockIdx.x;
    const long long stride = static_cast<long long>(gridDim.x) * gridDim.y * kThreads;
    for (long long i = cta * kThreads + threadIdx.x; i < total; i += stride) a.out[i] = 0.f;
    const int n_tiles = (a.H + kDownRows - 1) / kDownRows;
    for (long long i = cta * kThreads + threadIdx.x; i < n_tiles; i += stride) tile_count[i] = 0;
  }
  const bool report = blockIdx.x == 0;
  const Route r = route_slot(a, blockIdx.y, s, report);
  if (r.e < 0) return;
  const pw_block_entry ent = a.table[2 * r.e];
  if (ent.state != PW_PAGE_GPU) {
    if (report) latch_status(a.status, PW_ERR_PAGE_NOT_RESIDENT);
    return;
  }
  const int i0 = blockIdx.x * kPairsPerTile;
  switch (ent.q) {
    case 3: gateup_tile<3>(a, r, ent, i0, s, h_ws); break;
    case 4: gateup_tile<4>(a, r, ent, i0, s, h_ws); break;
    case 5: gateup_tile<5>(a, r, ent, i0, s, h_ws); break;
    case 6: gateup_tile<6>(a, r, ent, i0, s, h_ws); break;
    case 8: gateup_tile<8>(a, r, ent, i0, s, h_ws); break;
    default:
      if (report) latch_status(a.status, PW_ERR_UNSUPPORTED_Q);
  }
}

// ---------------------------------------------------------------- down

template <int Q, int R, int NT>
__device__ void down_group(const LayerArgs& a, const Route& r, const pw_block_entry& ent,
                           int n0, int g0, int nt, const SmemPtrs& s, const float* h_ws,
                           float* y_ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KW = a.I / 32;
  const int N = a.H;
  const long long plane_stride = static_cast<long long>(N) * KW;
  int row[R];
#pragma unroll
  for (int g = 0; g < R; ++g) row[g] = n0 + 32 * g + lane;
  int lo, hi;
  warp_range(KW, lo, hi);
  auto loader = [&](float* act, int c0, int cols) {
    const int c = lane * 4;
#pragma unroll
    for (int tk = 0; tk < NT; ++tk) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tk < nt && c < cols)
        v = *reinterpret_cast<const float4*>(h_ws + static_cast<long long>(r.off + g0 + tk) * a.I +
                                             c0 + c);
      *reinterpret_cast<float4*>(act + tk * kCC + c) = v;
    }
  };
  float acc[R][NT];
  rows_dot<Q, R, NT>(ent.planes, plane_stride, N, row, lo, hi, s, loader, acc);
#pragma unroll
  for (int tk = 0; tk < NT; ++tk)
#pragma unroll
    for (int g = 0; g < R; ++g) s.red[((warp * kTG + tk) * 2 + g) * 32 + lane] = acc[g][tk];
  __syncthreads();
  for (int i = threadIdx.x; i < 32 * R * nt; i += kThreads) {
    const int L = i & 31, g = (i >> 5) % R, tk = (i >> 5) / R;
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) y += s.red[((w * kTG + tk) * 2 + g) * 32 + L];
    y_ws[static_cast<long long>(s.pairs[g0 + tk]) * a.H + n0 + 32 * g + L] = y;
  }
  __syncthreads();
}

template <int Q, int R>
__device__ void down_tile(const LayerArgs& a, const Route& r, const pw_block_entry& ent, int n0,
                          const SmemPtrs& s, const float* h_ws, float* y_ws) {
  int row0[R];
#pragma unroll
  for (int g = 0; g < R; ++g) row0[g] = n0 + 32 * g;
  load_luts<Q, R>(ent.lut, row0, s);
  __syncthreads();
  for (int g0 = 0; g0 < r.ne; g0 += kTG) {
    const int nt = min(kTG, r.ne - g0);
    if (nt == 1) down_group<Q, R, 1>(a, r, ent, n0, g0, nt, s, h_ws, y_ws);
    else if (nt == 2) down_group<Q, R, 2>(a, r, ent, n0, g0, nt, s, h_ws, y_ws);
    else down_group<Q, R, 4>(a, r, ent, n0, g0, nt, s, h_ws, y_ws);
  }
}

template <int R>
__device__ void down_dispatch(const LayerArgs& a, const Route& r, const pw_block_entry& ent,
                              int n0, const SmemPtrs& s, const float* h_ws, float* y_ws) {
  switch (ent.q) {
    case 3: down_tile<3, R>(a, r, ent, n0, s, h_ws, y_ws); break;
    case 4: down_tile<4, R>(a, r, ent, n0, s, h_ws, y_ws); break;
    case 5: down_tile<5, R>(a, r, ent, n0, s, h_ws, y_ws); break;
    case 6: down_tile<6, R>(a, r, ent, n0, s, h_ws, y_ws); break;
    default: down_tile<8, R>(a, r, ent, n0, s, h_ws, y_ws); break;
  }
}

// Pairs of an expert that cannot be computed contribute zero.
__device__ void zero_pairs(const LayerArgs& a, const Route& r, int n0, int rows,
                           const SmemPtrs& s, float* y_ws) {
  for (int i = threadIdx.x; i < r.ne * rows; i += kThreads)
    y_ws[static_cast<long long>(s.pairs[i / rows]) * a.H + n0 + (i % rows)] = 0.f;
}

__global__ void __launch_bounds__(kThreads, 2) decode_down_kernel(const LayerArgs a, const float* h_ws,
                                                                  float* y_ws, int* tile_count) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const SmemPtrs s = carve(smem_raw);
  const Route r = route_slot(a, blockIdx.y, s, false);
  if (r.e < 0) return;
  const pw_block_entry gu = a.table[2 * r.e];
  const pw_block_entry ent = a.table[2 * r.e + 1];
  const bool report = blockIdx.x == 0;
  const int n0 = blockIdx.x * kDownRows;
  const int rows = min(kDownRows, a.H - n0);   // 64, or 32 on a ragged last tile
  if (gu.state != PW_PAGE_GPU || ent.state != PW_PAGE_GPU) {
    if (report) latch_status(a.status, PW_ERR_PAGE_NOT_RESIDENT);
    zero_pairs(a, r, n0, rows, s, y_ws);
  } else if (!supported_q(gu.q) || !supported_q(ent.q)) {
    if (report && !supported_q(ent.q)) latch_status(a.status, PW_ERR_UNSUPPORTED_Q);
    zero_pairs(a, r, n0, rows, s, y_ws);  // an unusable block: this expert contributes 0
  } else if (rows == kDownRows) {
    down_dispatch<2>(a, r, ent, n0, s, h_ws, y_ws);
  } else {
    down_dispatch<1>(a, r, ent, n0, s, h_ws, y_ws);
  }
  // Arrival: the last of the routed experts' CTAs on this row tile combines.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int n_routed = s.misc[3];
    const int old = atomicAdd(&tile_count[blockIdx.x], 1);
    s.misc[4] = (old == n_routed - 1);
    if (old == n_routed - 1) tile_count[blockIdx.x] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!s.misc[4]) return;
  __threadfence();
  for (int i = threadIdx.x; i < a.T * rows; i += kThreads) {
    const int t = i / rows, n = n0 + i % rows;
    float acc = 0.f;
    for (int j = 0; j < a.k; ++j) {
      const int p = t * a.k + j;
      const int e = a.topk_ids[p];
      if (e < 0 || e >= a.E) continue;
      acc = fmaf(a.topk_weights[p], __ldcg(y_ws + static_cast<long long>(p) * a.H + n), acc);
    }
    a.out[static_cast<long long>(t) * a.H + n] = acc;
  }
}

}  // namespace

int decode_max_pairs() { return kMaxPairs; }
int decode_max_experts() { return kMaxExperts; }

namespace {
size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}  // namespace

// Workspace: h [T*k][I] fp32 | y [T*k][H] fp32 | per-row-tile counters [H/32].
size_t decode_workspace_bytes(const pw_moe_shape& s) {
  const size_t pairs = static_cast<size_t>(s.T) * s.k;
  return round256(sizeof(float) * pairs * s.I) + round256(sizeof(float) * pairs * s.H) +
         round256(sizeof(int) * (s.H / 32));
}

cudaError_t launch_decode(const LayerArgs& a, void* ws, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int n_pairs = a.T * a.k;
  if (n_pairs == 0) return cudaSuccess;
  const int slots = min(a.E, n_pairs);
  char* base = static_cast<char*>(ws);
  float* h_ws = reinterpret_cast<float*>(base);
  base += round256(sizeof(float) * static_cast<size_t>(n_pairs) * a.I);
  float* y_ws = reinterpret_cast<float*>(base);
  base += round256(sizeof(float) * static_cast<size_t>(n_pairs) * a.H);
  int* tile_count = reinterpret_cast<int*>(base);
  decode_gateup_kernel<<<dim3(a.I / kPairsPerTile, slots), kThreads, kSmemBytes, stream>>>(
      a, h_ws, tile_count);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_down_kernel<<<dim3((a.H + kDownRows - 1) / kDownRows, slots), kThreads, kSmemBytes,
                       stream>>>(a, h_ws, y_ws, tile_count);
  return cudaGetLastError();
}

}  // namespace pw
