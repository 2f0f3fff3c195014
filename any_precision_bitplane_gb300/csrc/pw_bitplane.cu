// Overlay bitplane encoding and the top-b read-back.
//
// PagedWeight, "Core components" 1 (Paged Weight representation): weights are
// kept in Any-Precision's overlay bitplane format; a b-bit view of a block reads
// its top b planes.  Layout: uint32 [8][K/32][N], plane p = bit (7-p) of the
// code; word [p][w][n] holds columns 32w..32w+31 of row n, column 32w+t at bit t.
#include "pw_internal.cuh"

namespace pw {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// One warp encodes one 32-column word of one row: lane t holds the code of
// column 32w+t, and a ballot over bit (7-p) is exactly plane p's word.  Work
// item wi = w * N + n walks word columns so that consecutive warps write
// consecutive rows of a word column.
__global__ void __launch_bounds__(256) pack_bitplanes_kernel(const uint8_t* __restrict__ codes,
                                                             int N, int K,
                                                             uint32_t* __restrict__ planes) {
  const int lane = threadIdx.x & 31;
  const long long n_words = static_cast<long long>(N) * (K / 32);
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long wi = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       wi < n_words; wi += warps) {
    const long long w = wi / N, n = wi % N;
    const uint32_t c = codes[n * K + w * 32 + lane];
    uint32_t mine = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const uint32_t word = __ballot_sync(kFull, (c >> (7 - p)) & 1u);
      if (lane == p) mine = word;
    }
    if (lane < 8) planes[static_cast<long long>(lane) * n_words + wi] = mine;
  }
}

// One thread per output index: gather bit (k mod 32) of word k/32 of row n
// from the first b planes, plane 0 landing in the top index bit.
__global__ void __launch_bounds__(256) unpack_top_kernel(const uint32_t* __restrict__ planes,
                                                         int N, int K, int b,
                                                         uint8_t* __restrict__ idx) {
  const long long total = static_cast<long long>(N) * K;
  const long long n_words = total / 32;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long n = i / K;
    const int k = static_cast<int>(i % K);
    const long long word = static_cast<long long>(k >> 5) * N + n;
    const int bit = k & 31;
    uint32_t v = 0;
    for (int p = 0; p < b; ++p) v = (v << 1) | ((planes[p * n_words + word] >> bit) & 1u);
    idx[i] = static_cast<uint8_t>(v);
  }
}

int grid_for(long long work, int per_block, int cap) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_pack_bitplanes(const uint8_t* codes, int N, int K, uint32_t* planes,
                                  cudaStream_t s) {
  const long long n_words = static_cast<long long>(N) * (K / 32);
  if (n_words == 0) return cudaSuccess;
  pack_bitplanes_kernel<<<grid_for(n_words, 8, 64 * sm_count()), 256, 0, s>>>(codes, N, K, planes);
  return cudaGetLastError();
}

cudaError_t launch_unpack_top(const uint32_t* planes, int N, int K, int b, uint8_t* idx,
                              cudaStream_t s) {
  const long long total = static_cast<long long>(N) * K;
  if (total == 0) return cudaSuccess;
  unpack_top_kernel<<<grid_for(total, 256, 64 * sm_count()), 256, 0, s>>>(planes, N, K, b, idx);
  return cudaGetLastError();
}

}  // namespace pw
