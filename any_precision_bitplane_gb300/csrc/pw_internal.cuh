// Internal declarations shared by the libpw translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "pw.h"

struct pw_page_table {
  int32_t num_blocks;
  int device;
  pw_block_entry* d_entries;  // fixed device address for the table's lifetime
  int32_t* d_status;          // first device-side error latched by forward calls
  int32_t* stats_counts = nullptr;  // routing statistics (caller's buffers) or NULL
  float* stats_mass = nullptr;
};

namespace pw {

// ---- error reporting (host) ------------------------------------------------
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t err, const char* what);
void clear_error();

// ---- per-device state (host) -------------------------------------------------
// Everything cached on the host is keyed by the device ordinal, so calls on
// several devices of one process (each with that device current) each get
// their own set-up and SM count.  All of it is safe to call from several
// host threads.
constexpr int kMaxDevices = 64;
enum SetupKey { kSetupDecode = 0, kSetupGemm = 1, kSetupKeys = 2 };
// Ordinal of the current device (PW_OK), or an error status with a message.
int current_device(int* dev);
// SM count of the current device (at least 1).
int sm_count();
// Runs `fn` (kernel attribute set-up) once per (key, current device); later
// calls return cudaSuccess without running it.  A failure is not cached.
cudaError_t setup_once(SetupKey key, cudaError_t (*fn)());

// Checks shared by the forward entry points (pw_moe_forward[_path] and
// pw_moe_forward_noalloc): shape, table, pointers and alignment, and that the
// current device is an sm_103 device and the table's device.  Fills *a; sets
// *empty when the call has no tokens (nothing to launch).
struct LayerArgs;
int check_forward_args(const pw_moe_shape* shape, const void* hidden, const int32_t* topk_ids,
                       const float* topk_weights, const pw_page_table* table, float* out,
                       LayerArgs* a, bool* empty);

// ---- device helpers ----------------------------------------------------------
__device__ __forceinline__ void latch_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ bool supported_q(int q) {
  return q == 3 || q == 4 || q == 5 || q == 6 || q == 8;
}

inline bool supported_q_host(int q) { return q == 3 || q == 4 || q == 5 || q == 6 || q == 8; }

// ---- launchers (each returns the launch error) -----------------------------
cudaError_t launch_pack_bitplanes(const uint8_t* codes, int N, int K, uint32_t* planes,
                                  cudaStream_t s);
cudaError_t launch_unpack_top(const uint32_t* planes, int N, int K, int b, uint8_t* idx,
                              cudaStream_t s);
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids,
                              float* wts, cudaStream_t s);
// With `logits` (float [n_pairs / k][E]) the routing is fused in front of the
// grouping: ids (then written, [n_pairs]) and route_wts receive its output.
cudaError_t launch_permute(const int32_t* ids, int n_pairs, int E, int32_t* offsets,
                           int32_t* perm, int32_t* inv, int32_t* status, cudaStream_t s,
                           const float* logits = nullptr, int k = 1, float* route_wts = nullptr);

constexpr int kMaxCommitPerLaunch = 240;  // keeps the parameter block under 4 KB
struct CommitBatch {
  int32_t n;
  int32_t kind;  // 0 = bitwidth + LUT, 1 = planes + state
  int32_t ids[kMaxCommitPerLaunch];
  int32_t ival[kMaxCommitPerLaunch];
  const void* ptr[kMaxCommitPerLaunch];
};
cudaError_t launch_commit(pw_block_entry* entries, const CommitBatch& batch, cudaStream_t s);

// Measurement hook (pw_set_timing_events): events recorded around the
// dominant kernel of each forward call; record_timing is a no-op for NULL.
struct TimingEvents {
  cudaEvent_t before = nullptr;
  cudaEvent_t after = nullptr;
};
extern TimingEvents g_timing;
cudaError_t record_timing(cudaEvent_t ev, cudaStream_t s);

// Fused layer, decode path.
struct LayerArgs {
  int32_t T, H, I, E, k;
  const uint16_t* hidden;        // bf16 bits [T][H]
  const int32_t* topk_ids;       // [T][k]
  const float* topk_weights;     // [T][k]
  const pw_block_entry* table;   // [2E]
  float* out;                    // [T][H]
  int32_t* status;
  int32_t* stats_counts;         // [E] routing statistics to accumulate, or NULL
  float* stats_mass;             // [E]
  // Fused routing: with logits (float [T][E]) the launch that groups the
  // pairs first routes the tokens into route_ids / route_wts (which are then
  // topk_ids / topk_weights); NULL when the caller routed.
  const float* logits = nullptr;
  int32_t* route_ids = nullptr;
  float* route_wts = nullptr;
};
// Routing statistics of one call (pairs per expert, sum of their weights),
// added to a.stats_counts / a.stats_mass; no-op when they are NULL.
cudaError_t launch_routing_stats(const LayerArgs& a, cudaStream_t s);
// In decode calls of at least kHybridMinTokens tokens (when the shape allows
// it), experts with at least kHeavyMinTokens pairs go through the tensor-core
// GEMM kernels of the prefill path; the others through the decode kernels,
// which stream an expert's weights once per group of 4 tokens.  Smaller
// calls skip the GEMM launches (three of them) altogether.
constexpr int kHeavyMinTokens = 8;
constexpr int kHybridMinTokens = 16;
// `hybrid` = false keeps every expert on the decode kernels (and the
// workspace free of the GEMM path's buffers).
size_t decode_workspace_bytes(const pw_moe_shape& s, bool hybrid = true);
cudaError_t launch_decode(const LayerArgs& a, void* ws, cudaStream_t s, bool hybrid = true);
int decode_max_pairs();
int decode_max_experts();

// Fused layer, prefill path.
size_t prefill_workspace_bytes(const pw_moe_shape& s);
cudaError_t launch_prefill(const LayerArgs& a, void* ws, cudaStream_t s);
int prefill_min_pairs(const pw_moe_shape& s);
bool prefill_shape_ok(const pw_moe_shape& s);  // H % 128 == 0, I % 64 == 0, E <= 1024
// The GEMM kernels of the prefill path over the experts that hold at least
// min_tokens pairs, on a grouping (offsets, perm) made by the caller; writes
// y[pair][H] of those pairs.  Scratch: heavy_scratch_bytes(s).
size_t heavy_scratch_bytes(const pw_moe_shape& s);
cudaError_t launch_heavy(const LayerArgs& a, const int32_t* offsets, const int32_t* perm, float* y,
                         void* scratch, int min_tokens, cudaStream_t s);

// Bit-exact checks of the kernels' own index extraction and table lookups
// (pw_debug_index / pw_debug_dequant), and the byte ranges of a workspace a
// test may read back (pw_debug_workspace_section).
cudaError_t launch_index_check(const uint32_t* planes, int N, int K, int q, bool nibbles,
                               uint8_t* idx, cudaStream_t s);
cudaError_t launch_dequant_check(const uint32_t* planes, const uint16_t* lut, int N, int K, int q,
                                 float* out, int32_t* status, cudaStream_t s);
cudaError_t launch_half_index_check(const uint32_t* planes, int N, int K, int q, uint8_t* idx,
                                    cudaStream_t s);
cudaError_t launch_half_dequant_check(const uint32_t* planes, const uint16_t* lut, int N, int K,
                                      int q, float* out, cudaStream_t s);
int decode_ws_section(const pw_moe_shape& shape, int section, size_t* offset, size_t* bytes);
int prefill_ws_section(const pw_moe_shape& shape, int section, size_t* offset, size_t* bytes);

// Failure-detection checks (pw_debug_bounded_wait): one bounded device wait
// of the forward kernels run against something never released.
cudaError_t launch_wait_check_decode(int32_t* status, uint32_t polls, cudaStream_t s);
cudaError_t launch_wait_check_mbar(int32_t* status, uint32_t polls, cudaStream_t s);
// The GEMM trace (built with PW_TRACE): false when tracing is compiled out.
bool gemm_trace_read(void* host, size_t bytes, cudaError_t* err);
size_t gemm_trace_bytes();
// The decode gate_up trace (built with PW_TRACE): false when compiled out.
bool decode_trace_read(void* host, size_t bytes, cudaError_t* err);
size_t decode_trace_bytes();

}  // namespace pw
