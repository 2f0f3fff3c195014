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
//   down:   per (routed expert e, tile of 32 down rows): same bitplane/LUT
//           read at the down block's q, dot with h -> y for each of e's pairs
//           (workspace).  The last CTA to finish a row tile (a per-tile
//           arrival counter) combines out[t] = sum_j w_tj * y[t*k + j] over
//           the tile in j order, so the output is deterministic.
//
// Layout of work inside a CTA: lane L owns row (row0 + L) of the tile, so each
// lane reads its own row's LUT from a lane-private shared-memory column
// (entry v of lane L at word v*32 + L: bank L, never a conflict); the 8 warps
// split the K columns and their partial sums meet in shared memory.
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
constexpr int kRows = 32;           // rows (gate/up pairs, or down rows) per CTA
constexpr int kTokGroup = 8;        // tokens per pass over the weights
constexpr int kChunkWords = 8;      // columns staged per activation chunk: 256
constexpr int kChunkCols = kChunkWords * 32;
constexpr int kMaxPairs = 4096;     // T*k limit of this path
constexpr int kMaxExperts = 1024;

struct Smem {
  // sizes in 4-byte words
  static constexpr int count = kMaxExperts;
  static constexpr int pairs = kMaxPairs;
  static constexpr int misc = 8;
  static constexpr int lut = 2 * 256 * 32;
  static constexpr int act = kWarps * kTokGroup * kChunkCols;
  static constexpr int red = kWarps * kTokGroup * 2 * 32;
  static constexpr int total = count + pairs + misc + lut + act + red;
};
constexpr size_t kSmemBytes = sizeof(float) * Smem::total;

struct SmemPtrs {
  int* count;
  int* pairs;
  int* misc;
  float* lut;
  float* act;
  float* red;
};

__device__ __forceinline__ SmemPtrs carve(void* base) {
  SmemPtrs s;
  int* p = static_cast<int*>(base);
  s.count = p;
  p += Smem::count;
  s.pairs = p;
  p += Smem::pairs;
  s.misc = p;
  p += Smem::misc;
  s.lut = reinterpret_cast<float*>(p);
  s.act = s.lut + Smem::lut;
  s.red = s.act + Smem::act;
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

// Lane-private LUT columns for R row groups: s.lut[(g * 2^Q + v) * 32 + L] =
// LUT_Q[row0_g + L][v] as fp32.  Each thread moves 8 fp16 entries (16 bytes).
template <int Q, int R>
__device__ __forceinline__ void load_luts(const uint16_t* lut, const int (&row0)[R],
                                          const SmemPtrs& s) {
  constexpr int kEnt = 1 << Q;
  constexpr int kVecPerRow = kEnt / 8;
  for (int g = 0; g < R; ++g) {
    for (int i = threadIdx.x; i < kRows * kVecPerRow; i += kThreads) {
      const int L = i & 31, vec = i >> 5;
      const uint4 raw = *reinterpret_cast<const uint4*>(
          lut + static_cast<long long>(row0[g] + L) * kEnt + vec * 8);
      const __half* h = reinterpret_cast<const __half*>(&raw);
      float* dst = s.lut + (g * kEnt + vec * 8) * 32 + L;
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j * 32] = __half2float(h[j]);
    }
  }
}

// Partial dot products of this lane's R rows over the warp's column range,
// for NT tokens whose activations the loader stages per 256-column chunk.
template <int Q, int R, int NT, class Loader>
__device__ __forceinline__ void rows_dot(const uint32_t* planes, long long plane_stride,
                                         const int (&row)[R], int kw_lo, int kw_hi, int KW,
                                         const SmemPtrs& s, const Loader& load_chunk,
                                         float (&acc)[R][NT]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* act = s.act + warp * (kTokGroup * kChunkCols);
#pragma unroll
  for (int g = 0; g < R; ++g)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[g][t] = 0.f;
  for (int kw0 = kw_lo; kw0 < kw_hi; kw0 += kChunkWords) {
    const int nw = min(kChunkWords, kw_hi - kw0);
    __syncwarp();
    load_chunk(act, kw0 * 32, nw * 32);
    __syncwarp();
    for (int ww = 0; ww < nw; ++ww) {
      uint32_t pl[R][Q];
#pragma unroll
      for (int g = 0; g < R; ++g)
#pragma unroll
        for (int p = 0; p < Q; ++p)
          pl[g][p] = __ldg(planes + p * plane_stride + static_cast<long long>(row[g]) * KW + kw0 + ww);
      const float* a_col = act + ww * 32;
#pragma unroll 4
      for (int t = 0; t < 32; ++t) {
        float w[R];
#pragma unroll
        for (int g = 0; g < R; ++g) {
          uint32_t idx = 0;
#pragma unroll
          for (int p = 0; p < Q; ++p) idx = (idx << 1) | ((pl[g][p] >> t) & 1u);
          w[g] = s.lut[(g * (1 << Q) + idx) * 32 + lane];
        }
#pragma unroll
        for (int tk = 0; tk < NT; ++tk) {
          const float x = a_col[tk * kChunkCols + t];
#pragma unroll
          for (int g = 0; g < R; ++g) acc[g][tk] = fmaf(x, w[g], acc[g][tk]);
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
  const long long plane_stride = static_cast<long long>(2 * a.I) * KW;
  const int row[2] = {i0 + lane, a.I + i0 + lane};
  int lo, hi;
  warp_range(KW, lo, hi);
  auto loader = [&](float* act, int c0, int cols) {
    for (int tk = 0; tk < NT; ++tk) {
      const bool live = tk < nt;
      const int t = live ? s.pairs[g0 + tk] / a.k : 0;
      const uint16_t* src = a.hidden + static_cast<long long>(t) * a.H + c0;
      for (int c = lane * 8; c < cols; c += 256) {
        float v[8];
        if (live) {
          const uint4 raw = *reinterpret_cast<const uint4*>(src + c);
          const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = bf16_bits_to_float(h[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = 0.f;
        }
        float4* d = reinterpret_cast<float4*>(act + tk * kChunkCols + c);
        d[0] = make_float4(v[0], v[1], v[2], v[3]);
        d[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  };
  float acc[2][NT];
  rows_dot<Q, 2, NT>(ent.planes, plane_stride, row, lo, hi, KW, s, loader, acc);
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) {
    s.red[((warp * kTokGroup + tk) * 2 + 0) * 32 + lane] = acc[0][tk];
    s.red[((warp * kTokGroup + tk) * 2 + 1) * 32 + lane] = acc[1][tk];
  }
  __syncthreads();
  if (threadIdx.x < 32 * nt) {
    const int tk = threadIdx.x >> 5;
    float g = 0.f, u = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      g += s.red[((w * kTokGroup + tk) * 2 + 0) * 32 + lane];
      u += s.red[((w * kTokGroup + tk) * 2 + 1) * 32 + lane];
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
  for (int g0 = 0; g0 < r.ne; g0 += kTokGroup) {
    const int nt = min(kTokGroup, r.ne - g0);
    if (nt == 1) gateup_group<Q, 1>(a, r, ent, i0, g0, nt, s, h_ws);
    else if (nt == 2) gateup_group<Q, 2>(a, r, ent, i0, g0, nt, s, h_ws);
    else if (nt <= 4) gateup_group<Q, 4>(a, r, ent, i0, g0, nt, s, h_ws);
    else gateup_group<Q, 8>(a, r, ent, i0, g0, nt, s, h_ws);
  }
}

__global__ void __launch_bounds__(kThreads, 1) decode_gateup_kernel(const LayerArgs a, float* h_ws,
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
    for (long long i = cta * kThreads + threadIdx.x; i < a.H / kRows; i += stride) tile_count[i] = 0;
  }
  const bool report = blockIdx.x == 0;
  const Route r = route_slot(a, blockIdx.y, s, report);
  if (r.e < 0) return;
  const pw_block_entry ent = a.table[2 * r.e];
  if (ent.state != PW_PAGE_GPU) {
    if (report) latch_status(a.status, PW_ERR_PAGE_NOT_RESIDENT);
    return;
  }
  const int i0 = blockIdx.x * kRows;
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

template <int Q, int NT>
__device__ void down_group(const LayerArgs& a, const Route& r, const pw_block_entry& ent,
                           int n0, int g0, int nt, const SmemPtrs& s, const float* h_ws,
                           float* y_ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KW = a.I / 32;
  const long long plane_stride = static_cast<long long>(a.H) * KW;
  const int row[1] = {n0 + lane};
  int lo, hi;
  warp_range(KW, lo, hi);
  auto loader = [&](float* act, int c0, int cols) {
    for (int tk = 0; tk < NT; ++tk) {
      const bool live = tk < nt;
      const float* src = h_ws + static_cast<long long>(r.off + g0 + (live ? tk : 0)) * a.I + c0;
      for (int c = lane * 8; c < cols; c += 256) {
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (live) {
          v0 = *reinterpret_cast<const float4*>(src + c);
          v1 = *reinterpret_cast<const float4*>(src + c + 4);
        }
        float4* d = reinterpret_cast<float4*>(act + tk * kChunkCols + c);
        d[0] = v0;
        d[1] = v1;
      }
    }
  };
  float acc[1][NT];
  rows_dot<Q, 1, NT>(ent.planes, plane_stride, row, lo, hi, KW, s, loader, acc);
#pragma unroll
  for (int tk = 0; tk < NT; ++tk) s.red[((warp * kTokGroup + tk) * 2) * 32 + lane] = acc[0][tk];
  __syncthreads();
  if (threadIdx.x < 32 * nt) {
    const int tk = threadIdx.x >> 5;
    float y = 0.f;
    for (int w = 0; w < kWarps; ++w) y += s.red[((w * kTokGroup + tk) * 2) * 32 + lane];
    y_ws[static_cast<long long>(s.pairs[g0 + tk]) * a.H + n0 + lane] = y;
  }
  __syncthreads();
}

template <int Q>
__device__ void down_tile(const LayerArgs& a, const Route& r, const pw_block_entry& ent, int n0,
                          const SmemPtrs& s, const float* h_ws, float* y_ws) {
  const int row0[1] = {n0};
  load_luts<Q, 1>(ent.lut, row0, s);
  __syncthreads();
  for (int g0 = 0; g0 < r.ne; g0 += kTokGroup) {
    const int nt = min(kTokGroup, r.ne - g0);
    if (nt == 1) down_group<Q, 1>(a, r, ent, n0, g0, nt, s, h_ws, y_ws);
    else if (nt == 2) down_group<Q, 2>(a, r, ent, n0, g0, nt, s, h_ws, y_ws);
    else if (nt <= 4) down_group<Q, 4>(a, r, ent, n0, g0, nt, s, h_ws, y_ws);
    else down_group<Q, 8>(a, r, ent, n0, g0, nt, s, h_ws, y_ws);
  }
}

// Pairs of an expert that cannot be computed contribute zero.
__device__ void zero_pairs(const LayerArgs& a, const Route& r, int n0, const SmemPtrs& s,
                           float* y_ws) {
  for (int i = threadIdx.x; i < r.ne * 32; i += kThreads)
    y_ws[static_cast<long long>(s.pairs[i >> 5]) * a.H + n0 + (i & 31)] = 0.f;
}

__global__ void __launch_bounds__(kThreads, 1) decode_down_kernel(const LayerArgs a, const float* h_ws,
                                                                  float* y_ws, int* tile_count) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const SmemPtrs s = carve(smem_raw);
  const Route r = route_slot(a, blockIdx.y, s, false);
  if (r.e < 0) return;
  const pw_block_entry gu = a.table[2 * r.e];
  const pw_block_entry ent = a.table[2 * r.e + 1];
  const bool report = blockIdx.x == 0;
  const int n0 = blockIdx.x * kRows;
  if (gu.state != PW_PAGE_GPU || ent.state != PW_PAGE_GPU) {
    if (report) latch_status(a.status, PW_ERR_PAGE_NOT_RESIDENT);
    zero_pairs(a, r, n0, s, y_ws);
  } else if (!supported_q(gu.q)) {
    zero_pairs(a, r, n0, s, y_ws);  // gate_up skipped this expert; h is not valid
  } else {
    switch (ent.q) {
      case 3: down_tile<3>(a, r, ent, n0, s, h_ws, y_ws); break;
      case 4: down_tile<4>(a, r, ent, n0, s, h_ws, y_ws); break;
      case 5: down_tile<5>(a, r, ent, n0, s, h_ws, y_ws); break;
      case 6: down_tile<6>(a, r, ent, n0, s, h_ws, y_ws); break;
      case 8: down_tile<8>(a, r, ent, n0, s, h_ws, y_ws); break;
      default:
        if (report) latch_status(a.status, PW_ERR_UNSUPPORTED_Q);
        zero_pairs(a, r, n0, s, y_ws);
    }
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
  const int lane = threadIdx.x & 31;
  for (int t = threadIdx.x >> 5; t < a.T; t += kWarps) {
    float acc = 0.f;
    for (int j = 0; j < a.k; ++j) {
      const int p = t * a.k + j;
      const int e = a.topk_ids[p];
      if (e < 0 || e >= a.E) continue;
      acc = fmaf(a.topk_weights[p], __ldcg(y_ws + static_cast<long long>(p) * a.H + n0 + lane), acc);
    }
    a.out[static_cast<long long>(t) * a.H + n0 + lane] = acc;
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
         round256(sizeof(int) * (s.H / kRows));
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
  decode_gateup_kernel<<<dim3(a.I / kRows, slots), kThreads, kSmemBytes, stream>>>(a, h_ws,
                                                                                   tile_count);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_down_kernel<<<dim3(a.H / kRows, slots), kThreads, kSmemBytes, stream>>>(a, h_ws, y_ws,
                                                                                 tile_count);
  return cudaGetLastError();
}

}  // namespace pw
