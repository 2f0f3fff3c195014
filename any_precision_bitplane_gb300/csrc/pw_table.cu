// Stream-ordered updates of the Weight Page Table.
//
// PagedWeight, "Core components" 1 (Weight Page Table: committed bitwidth q_i
// and page state per block) and 3 (commits take effect only at a safe
// boundary).  The update list travels in the kernel's parameter block, so an
// update is one launch with no host-to-device copy and it is ordered on the
// stream like any other kernel: forward calls enqueued before it read the old
// entries, calls enqueued after it read the new ones.
#include "pw_internal.cuh"

namespace pw {
namespace {

__global__ void commit_kernel(pw_block_entry* __restrict__ entries, const CommitBatch batch) {
  for (int i = threadIdx.x; i < batch.n; i += blockDim.x) {
    pw_block_entry& ent = entries[batch.ids[i]];
    if (batch.kind == 0) {
      ent.q = batch.ival[i];
      ent.lut = static_cast<const uint16_t*>(batch.ptr[i]);
    } else {
      ent.planes = static_cast<const uint32_t*>(batch.ptr[i]);
      ent.state = batch.ival[i];
    }
  }
}

}  // namespace

cudaError_t launch_commit(pw_block_entry* entries, const CommitBatch& batch, cudaStream_t s) {
  if (batch.n == 0) return cudaSuccess;
  commit_kernel<<<1, 256, 0, s>>>(entries, batch);
  return cudaGetLastError();
}

}  // namespace pw
