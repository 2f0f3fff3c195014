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
  // the same argument checks as pw_moe_forward, including that the current
  // device is the table's device (so the scratch address below is that
  // device's copy of the array)
  pw::LayerArgs a;
  bool empty = false;
  int rc = pw::check_forward_args(shape, hidden, topk_ids, topk_weights, table, out, &a, &empty);
  if (rc || empty) return rc;
  const pw_moe_shape& s = *shape;
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
  if ((rc = pw::current_device(&dev))) return rc;
  void* scratch = nullptr;
  if ((rc = pw::static_scratch_address(dev, &scratch))) return rc;
  cudaError_t e = pw::launch_decode(a, scratch, stream, false);
  if (e != cudaSuccess) return pw::cuda_fail(e, "forward launch");
  return PW_OK;
}
