// Router (softmax top-k with renormalised weights) and the token-to-expert
// permutation that groups (token, expert) pairs by expert.
#include <cfloat>
#include <climits>

#include "pw_internal.cuh"
#include "pw_router.cuh"

namespace pw {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// One warp per token (route_token_warp).
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits,
                                                         int T, int E, int k,
                                                         int32_t* __restrict__ ids,
                                                         float* __restrict__ wts) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  route_token_warp(logits + static_cast<long long>(t) * E, E, k, ids + static_cast<long long>(t) * k,
                   wts + static_cast<long long>(t) * k);
}

// Single CTA of 32 warps; warp w owns the contiguous run of pairs
// [w*L, (w+1)*L), L = ceil(n_pairs / 32).  Pass 1: each warp counts its
// pairs per expert (__match_any_sync groups same-expert lanes; the group's
// first lane adds the group size to the warp's own row of counts, so no
// atomics).  Then thread e turns column e of the counts into the expert's
// running start per warp, and a block scan of the per-expert totals gives
// offsets.  Pass 2: each warp walks its run again and places every pair at
// its warp's running start for the expert plus its rank among same-expert
// lanes of the step.  Runs are in pair order and ranks follow lane order, so
// the placement is the stable one: position = offsets[e] + earlier pairs of e.
constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

//
// With `logits` the routing is fused in front: the warps route the tokens
// (token t on warp t % 32) into ids / wts, which the rest then reads.
__global__ void __launch_bounds__(kPermThreads) permute_kernel(const int32_t* __restrict__ ids,
                                                               int n_pairs, int E,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ perm,
                                                               int32_t* __restrict__ inv,
                                                               int32_t* status,
                                                               const float* __restrict__ logits,
                                                               int k, int32_t* route_ids,
                                                               float* route_wts) {
  extern __shared__ int smem[];
  if (logits != nullptr) {
    const int T = n_pairs / k;
    for (int t = threadIdx.x >> 5; t < T; t += kPermWarps)
      route_token_warp(logits + static_cast<long long>(t) * E, E, k,
                       route_ids + static_cast<long long>(t) * k, route_wts + static_cast<long long>(t) * k);
    __syncthreads();   // the routed ids are visible to the whole CTA
  }
  int* s_cnt = smem;                   // [kPermWarps][E]: counts, then running starts
  __shared__ int s_warp_sum[kPermWarps];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int L = (n_pairs + kPermWarps - 1) / kPermWarps;
  const int lo = min(n_pairs, warp * L), hi = min(n_pairs, lo + L);

  for (int i = tid; i < kPermWarps * E; i += kPermThreads) s_cnt[i] = 0;
  __syncthreads();
  int* my = s_cnt + warp * E;
  for (int base = lo; base < hi; base += 32) {
    const int p = base + lane;
    const int e = (p < hi) ? ids[p] : -1;
    const bool valid = (e >= 0 && e < E);
    if (p < hi && !valid) latch_status(status, PW_ERR_BAD_EXPERT_ID);
    const unsigned peers = __match_any_sync(kFull, valid ? e : -1);
    if (valid && (peers & ((1u << lane) - 1u)) == 0) my[e] += __popc(peers);
  }
  __syncthreads();

  // column e: per-warp exclusive prefix (in place) and the expert's total
  int tot = 0;
  if (tid < E) {
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = s_cnt[w * E + tid];
      s_cnt[w * E + tid] = tot;
      tot += c;
    }
  }
  // exclusive block scan of the totals over experts (thread e holds expert e)
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp_sum[warp] = incl;
  __syncthreads();
  int before = incl - tot;
  for (int w = 0; w < warp; ++w) before += s_warp_sum[w];
  if (tid < E) {
    offsets[tid] = before;
    for (int w = 0; w < kPermWarps; ++w) s_cnt[w * E + tid] += before;
  }
  if (tid == kPermThreads - 1) {
    int total = 0;
    for (int w = 0; w < kPermWarps; ++w) total += s_warp_sum[w];
    offsets[E] = total;
  }
  __syncthreads();

  for (int base = lo; base < hi; base += 32) {
    const int p = base + lane;
    const int e = (p < hi) ? ids[p] : -1;
    const bool valid = (e >= 0 && e < E);
    const unsigned peers = __match_any_sync(kFull, valid ? e : -1);
    const unsigned lower = peers & ((1u << lane) - 1u);
    int pos = -1;
    if (valid) {
      pos = my[e] + __popc(lower);
      perm[pos] = p;
    }
    if (p < hi && inv != nullptr) inv[p] = pos;
    __syncwarp();   // every lane has read its start before the group's first lane moves it
    if (valid && lower == 0) my[e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids,
                              float* wts, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + 7) / 8;
  route_topk_kernel<<<blocks, 256, 0, s>>>(logits, T, E, k, ids, wts);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* ids, int n_pairs, int E, int32_t* offsets,
                           int32_t* perm, int32_t* inv, int32_t* status, cudaStream_t s,
                           const float* logits, int k, float* route_wts) {
  const size_t smem = sizeof(int) * static_cast<size_t>(E) * kPermWarps;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  permute_kernel<<<1, kPermThreads, smem, s>>>(ids, n_pairs, E, offsets, perm, inv, status, logits, k,
                                               const_cast<int32_t*>(ids), route_wts);
  return cudaGetLastError();
}

namespace {

__global__ void __launch_bounds__(256) routing_stats_kernel(const int32_t* __restrict__ ids,
                                                            const float* __restrict__ wts,
                                                            int n_pairs, int E,
                                                            int32_t* __restrict__ counts,
                                                            float* __restrict__ mass) {
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_pairs; p += gridDim.x * blockDim.x) {
    const int e = ids[p];
    if (e < 0 || e >= E) continue;
    atomicAdd(&counts[e], 1);
    atomicAdd(&mass[e], wts[p]);
  }
}

}  // namespace

cudaError_t launch_routing_stats(const LayerArgs& a, cudaStream_t s) {
  if (a.stats_counts == nullptr) return cudaSuccess;
  const int n_pairs = a.T * a.k;
  if (n_pairs == 0) return cudaSuccess;
  const int blocks = (n_pairs + 255) / 256 < 1024 ? (n_pairs + 255) / 256 : 1024;
  routing_stats_kernel<<<blocks, 256, 0, s>>>(a.topk_ids, a.topk_weights, n_pairs, a.E,
                                              a.stats_counts, a.stats_mass);
  return cudaGetLastError();
}

}  // namespace pw
