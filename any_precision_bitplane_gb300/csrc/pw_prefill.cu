// Fused mixed-precision MoE layer, prefill path (many tokens per expert).
#include <climits>

#include "pw_internal.cuh"

namespace pw {

size_t prefill_workspace_bytes(const pw_moe_shape&) { return 0; }

int prefill_min_pairs(const pw_moe_shape&) { return INT_MAX; }

cudaError_t launch_prefill(const LayerArgs&, void*, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pw
