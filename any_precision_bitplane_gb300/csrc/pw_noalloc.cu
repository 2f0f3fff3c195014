// pw_moe_forward_noalloc: the decode path of the fused layer for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin whose enqueue hook
// is handed only its input and output buffers, a runtime that fixes its memory
// budget at start-up and forbids allocation afterwards, or code running where
// a cudaMalloc would synchronise the device or break a capture.  For them the
// scratch the decode kernels need (per-pair gate/up activations, per-pair
// expert outputs and the per-tile arrival counters) lives in one file-scope
// device array of fixed size instead of a caller-provided workspace.
//
// The array is a static __device__ symbol: every GPU that loads libpw holds
// its kStaticScratchBytes until the process exits.  Host code cannot use the
// symbol's name as a device address, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current, on the
// first call made on it.
#include <cstdio>
#include <mutex>

#include "pw_internal.cuh"

namespace pw {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on device `dev` (which must be current).
int static_scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices)
    return fail(PW_ERR_INVALID_ARG, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    if (p == nullptr) return fail(PW_ERR_CUDA, "cudaGetSymbolAddress returned NULL");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PW_OK;
}

}  // namespace
}  // namespace pw

extern "C" int pw_moe_forward_noalloc(const pw_moe_shape* shape, const void* hidden,
                                      const int32_t* topk_ids, const float* topk_weights,
                                      const pw_page_table* table, float* out,
                                      cudaStream_t stream) {
  using pw::fail;
  if (shape == nullptr) return fail(PW_ERR_INVALID_ARG, "shape is NULL");
  const pw_moe_shape& s = *shape;
  if (s.T < 0 || s.H <= 0 || s.I <= 0 || s.E <= 0 || s.k <= 0)
    return fail(PW_ERR_INVALID_ARG, "shape has a non-positive size (T=%d H=%d I=%d E=%d k=%d)",
                s.T, s.H, s.I, s.E, s.k);
  if (s.H % 32 || s.I % 32)
    return fail(PW_ERR_SHAPE, "H (%d) and I (%d) must be multiples of 32", s.H, s.I);
  if (s.k > s.E) return fail(PW_ERR_SHAPE, "k (%d) > E (%d)", s.k, s.E);
  if (table == nullptr) return fail(PW_ERR_INVALID_ARG, "table is NULL");
  if (table->num_blocks != 2 * s.E)
    return fail(PW_ERR_SHAPE, "page table has %d blocks, shape needs 2E = %d", table->num_blocks,
                2 * s.E);
  if (s.T == 0) return PW_OK;
  if (!hidden || !topk_ids || !topk_weights || !out)
    return fail(PW_ERR_INVALID_ARG, "hidden, topk_ids, topk_weights and out must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(PW_ERR_INVALID_ARG, "hidden and out must be 16-byte aligned");
  const long long n_pairs = static_cast<long long>(s.T) * s.k;
  if (n_pairs > pw::decode_max_pairs() || s.E > pw::decode_max_experts())
    return fail(PW_ERR_SHAPE, "decode path limits: T*k <= %d, E <= %d", pw::decode_max_pairs(),
                pw::decode_max_experts());
  const size_t need = pw::decode_workspace_bytes(s, false);
  if (need > pw::kStaticScratchBytes)
    return fail(PW_ERR_WORKSPACE,
                "shape needs %zu bytes of scratch; the static scratch of "
                "pw_moe_forward_noalloc holds %zu bytes (use pw_moe_forward with a workspace)",
                need, pw::kStaticScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pw::cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return pw::cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(PW_ERR_UNSUPPORTED_DEVICE, "device %d is sm_%d%d; libpw is built for sm_103a", dev,
                major, minor);
  void* scratch = nullptr;
  int rc = pw::static_scratch_address(dev, &scratch);
  if (rc) return rc;
  pw::LayerArgs a;
  a.T = s.T;
  a.H = s.H;
  a.I = s.I;
  a.E = s.E;
  a.k = s.k;
  a.hidden = static_cast<const uint16_t*>(hidden);
  a.topk_ids = topk_ids;
  a.topk_weights = topk_weights;
  a.table = table->d_entries;
  a.out = out;
  a.status = table->d_status;
  a.stats_counts = table->stats_counts;
  a.stats_mass = table->stats_mass;
  e = pw::launch_decode(a, scratch, stream, false);
  if (e != cudaSuccess) return pw::cuda_fail(e, "forward launch");
  return PW_OK;
}
