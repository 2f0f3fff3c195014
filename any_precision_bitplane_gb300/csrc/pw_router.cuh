// Router of one token, run by one warp: softmax over E logits, the top k
// experts (ties to the lower id), the kept probabilities renormalised.  Used
// by the standalone router launch and, fused, by the launches that group the
// pairs (the decode prep and the prefill permutation).
#pragma once

#include <cfloat>
#include <climits>
#include <cstdint>

namespace pw {

// Lane l owns experts l, l+32, ... (E <= 1024, so one 32-bit mask per lane
// marks the experts already taken).  Each of the k rounds is a warp argmax by
// (logit descending, id ascending); softmax is monotone, so selecting on
// logits selects on probabilities.  The kept weights are the softmax over the
// kept logits, which equals the full softmax renormalised.  Lanes j < k write
// ids[j] and wts[j].  Every lane of the warp must call it.
__device__ __forceinline__ void route_token_warp(const float* __restrict__ row, int E, int k,
                                                 int32_t* __restrict__ ids,
                                                 float* __restrict__ wts) {
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;
  int my_e = -1;
  float my_v = -INFINITY;
  for (int r = 0; r < k; ++r) {
    float best_v = -INFINITY;
    int best_e = INT_MAX;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if ((taken >> i) & 1u) continue;
      const float v = row[e];
      if (v > best_v || (v == best_v && e < best_e)) {
        best_v = v;
        best_e = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(kAll, best_v, off);
      const int oe = __shfl_xor_sync(kAll, best_e, off);
      if (ov > best_v || (ov == best_v && oe < best_e)) {
        best_v = ov;
        best_e = oe;
      }
    }
    if (best_e == INT_MAX) best_e = -1;  // only NaN logits left
    if (best_e >= 0 && (best_e & 31) == lane) taken |= 1u << (best_e >> 5);
    if (lane == r) {
      my_e = best_e;
      my_v = best_v;
    }
  }
  const float top = __shfl_sync(kAll, my_v, 0);
  const float ex = (lane < k && my_e >= 0) ? expf(my_v - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kAll, sum, off);
  if (lane < k) {
    ids[lane] = my_e;
    wts[lane] = ex / sum;
  }
}

}  // namespace pw
