// extern "C" entry points of libpw: argument validation and launches only.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "pw_internal.cuh"

namespace pw {

TimingEvents g_timing;

cudaError_t record_timing(cudaEvent_t ev, cudaStream_t s) {
  if (ev == nullptr) return cudaSuccess;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &st);
  if (e != cudaSuccess) return e;
  return st == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, s);
}

namespace {
thread_local char g_err[512] = "";

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The kernels are built for sm_103a only; refuse other devices with a clear
// error instead of a launch failure.
int check_device() {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  static std::atomic<int> checked[kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
  if (checked[dev].load(std::memory_order_relaxed) == 1) return PW_OK;
  int major = 0, minor = 0;
  cudaError_t e;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  const bool ok = (major == 10 && minor == 3);
  checked[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  if (!ok)
    return fail(PW_ERR_UNSUPPORTED_DEVICE, "device %d is sm_%d%d; libpw is built for sm_103a", dev,
                major, minor);
  return PW_OK;
}

int check_shape(const pw_moe_shape* s) {
  if (s == nullptr) return fail(PW_ERR_INVALID_ARG, "shape is NULL");
  if (s->T < 0 || s->H <= 0 || s->I <= 0 || s->E <= 0 || s->k <= 0)
    return fail(PW_ERR_INVALID_ARG, "shape has a non-positive size (T=%d H=%d I=%d E=%d k=%d)",
                s->T, s->H, s->I, s->E, s->k);
  if (s->H % 32 || s->I % 32)
    return fail(PW_ERR_SHAPE, "H (%d) and I (%d) must be multiples of 32", s->H, s->I);
  if (s->k > s->E) return fail(PW_ERR_SHAPE, "k (%d) > E (%d)", s->k, s->E);
  if (static_cast<long long>(s->T) * s->k > (1LL << 30))
    return fail(PW_ERR_SHAPE, "T*k too large");
  return PW_OK;
}

int forward_impl(const pw_moe_shape* shape, const void* hidden, const int32_t* topk_ids,
                 const float* topk_weights, const pw_page_table* table, float* out,
                 void* workspace, size_t workspace_bytes, int32_t path, cudaStream_t stream,
                 const float* logits = nullptr) {
  if (path < PW_PATH_AUTO || path > PW_PATH_PREFILL)
    return fail(PW_ERR_INVALID_ARG, "unknown path %d", path);
  LayerArgs a;
  bool empty = false;
  int rc = check_forward_args(shape, hidden, topk_ids, topk_weights, table, out, &a, &empty);
  if (rc || empty) return rc;
  const pw_moe_shape& s = *shape;
  if (logits != nullptr) {
    if (!aligned(logits, 4)) return fail(PW_ERR_INVALID_ARG, "logits must be 4-byte aligned");
    if (s.E > 1024 || s.k > 32)
      return fail(PW_ERR_SHAPE, "the fused router needs E <= 1024 and k <= 32");
    a.logits = logits;
    a.route_ids = const_cast<int32_t*>(topk_ids);
    a.route_wts = const_cast<float*>(topk_weights);
  }
  const long long n_pairs = static_cast<long long>(s.T) * s.k;
  if (path == PW_PATH_AUTO) path = (n_pairs >= prefill_min_pairs(s)) ? PW_PATH_PREFILL : PW_PATH_DECODE;
  size_t need = (path == PW_PATH_DECODE) ? decode_workspace_bytes(s) : prefill_workspace_bytes(s);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return fail(PW_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes (got %zu)",
                need, workspace_bytes);
  cudaError_t e;
  if (path == PW_PATH_DECODE) {
    if (n_pairs > decode_max_pairs() || s.E > decode_max_experts())
      return fail(PW_ERR_SHAPE, "decode path limits: T*k <= %d, E <= %d", decode_max_pairs(),
                  decode_max_experts());
    e = launch_decode(a, workspace, stream);
  } else {
    if (!prefill_shape_ok(s))
      return fail(PW_ERR_SHAPE, "prefill path needs H %% 128 == 0, I %% 64 == 0 and E <= 1024");
    e = launch_prefill(a, workspace, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return PW_OK;
}

int update_table(pw_page_table* t, int32_t n, const int32_t* ids, int kind, const int32_t* ival,
                 const void* const* ptrs, cudaStream_t stream) {
  if (t == nullptr) return fail(PW_ERR_INVALID_ARG, "table is NULL");
  if (n < 0) return fail(PW_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return PW_OK;
  if (!ids || !ival || !ptrs) return fail(PW_ERR_INVALID_ARG, "NULL list");
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= t->num_blocks)
      return fail(PW_ERR_INVALID_ARG, "block id %d out of range [0, %d)", ids[i], t->num_blocks);
    if (kind == 0 && !supported_q_host(ival[i]))
      return fail(PW_ERR_UNSUPPORTED_Q, "q = %d is not in {3,4,5,6,8}", ival[i]);
    if (kind == 1 && (ival[i] < PW_PAGE_GPU || ival[i] > PW_PAGE_IN_TRANSFER))
      return fail(PW_ERR_INVALID_ARG, "page state %d unknown", ival[i]);
    if (ptrs[i] == nullptr || !aligned(ptrs[i], 16))
      return fail(PW_ERR_INVALID_ARG, "entry %d: pointer NULL or not 16-byte aligned", i);
  }
  int cur = 0;
  int rc = current_device(&cur);
  if (rc) return rc;
  cudaError_t e;
  if (cur != t->device)
    return fail(PW_ERR_INVALID_ARG, "current device %d is not the table's device %d", cur,
                t->device);
  for (int i0 = 0; i0 < n; i0 += kMaxCommitPerLaunch) {
    CommitBatch b;
    b.n = (n - i0 < kMaxCommitPerLaunch) ? n - i0 : kMaxCommitPerLaunch;
    b.kind = kind;
    for (int i = 0; i < b.n; ++i) {
      b.ids[i] = ids[i0 + i];
      b.ival[i] = ival[i0 + i];
      b.ptr[i] = ptrs[i0 + i];
    }
    e = launch_commit(t->d_entries, b, stream);
    if (e != cudaSuccess) return cuda_fail(e, "page table update");
  }
  return PW_OK;
}

}  // namespace

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t err, const char* what) {
  return fail(PW_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
}

void clear_error() { g_err[0] = 0; }

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices)
    return fail(PW_ERR_INVALID_ARG, "device ordinal %d outside 0..%d", *dev, kMaxDevices - 1);
  return PW_OK;
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t setup_once(SetupKey key, cudaError_t (*fn)()) {
  static std::atomic<bool> done[kMaxDevices][kSetupKeys];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev][key].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev][key].load(std::memory_order_relaxed)) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess) done[dev][key].store(true, std::memory_order_release);
  return e;
}

int check_forward_args(const pw_moe_shape* shape, const void* hidden, const int32_t* topk_ids,
                       const float* topk_weights, const pw_page_table* table, float* out,
                       LayerArgs* a, bool* empty) {
  *empty = false;
  int rc = check_shape(shape);
  if (rc) return rc;
  const pw_moe_shape& s = *shape;
  if (table == nullptr) return fail(PW_ERR_INVALID_ARG, "table is NULL");
  if (table->num_blocks != 2 * s.E)
    return fail(PW_ERR_SHAPE, "page table has %d blocks, shape needs 2E = %d", table->num_blocks,
                2 * s.E);
  if (s.T == 0) {
    *empty = true;
    return PW_OK;
  }
  if (!hidden || !topk_ids || !topk_weights || !out)
    return fail(PW_ERR_INVALID_ARG, "hidden, topk_ids, topk_weights and out must be non-NULL");
  if (!aligned(hidden, 16) || !aligned(out, 16))
    return fail(PW_ERR_INVALID_ARG, "hidden and out must be 16-byte aligned");
  if (!aligned(topk_ids, 4) || !aligned(topk_weights, 4))
    return fail(PW_ERR_INVALID_ARG, "topk_ids and topk_weights must be 4-byte aligned");
  if ((rc = check_device())) return rc;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  if (dev != table->device)
    return fail(PW_ERR_INVALID_ARG, "current device %d is not the page table's device %d", dev,
                table->device);
  a->T = s.T;
  a->H = s.H;
  a->I = s.I;
  a->E = s.E;
  a->k = s.k;
  a->hidden = static_cast<const uint16_t*>(hidden);
  a->topk_ids = topk_ids;
  a->topk_weights = topk_weights;
  a->table = table->d_entries;
  a->out = out;
  a->status = table->d_status;
  a->stats_counts = table->stats_counts;
  a->stats_mass = table->stats_mass;
  return PW_OK;
}

}  // namespace pw

using pw::fail;
using pw::cuda_fail;

extern "C" {

const char* pw_last_error(void) { return pw::g_err; }

int pw_version(void) { return 100; }

int pw_set_timing_events(cudaEvent_t before, cudaEvent_t after) {
  if ((before == nullptr) != (after == nullptr))
    return fail(PW_ERR_INVALID_ARG, "pass both events or neither");
  pw::g_timing.before = before;
  pw::g_timing.after = after;
  return PW_OK;
}

int pw_pack_bitplanes(const uint8_t* codes, int32_t N, int32_t K, uint32_t* planes,
                      cudaStream_t stream) {
  if (N < 0) return fail(PW_ERR_INVALID_ARG, "N < 0");
  if (K <= 0 || K % 32) return fail(PW_ERR_SHAPE, "K (%d) must be a positive multiple of 32", K);
  if (N == 0) return PW_OK;
  if (!codes || !planes) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  int rc = pw::check_device();
  if (rc) return rc;
  cudaError_t e = pw::launch_pack_bitplanes(codes, N, K, planes, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "pack launch");
}

int pw_unpack_top(const uint32_t* planes, int32_t N, int32_t K, int32_t b, uint8_t* idx,
                  cudaStream_t stream) {
  if (N < 0) return fail(PW_ERR_INVALID_ARG, "N < 0");
  if (K <= 0 || K % 32) return fail(PW_ERR_SHAPE, "K (%d) must be a positive multiple of 32", K);
  if (b < 1 || b > 8) return fail(PW_ERR_UNSUPPORTED_Q, "b = %d not in 1..8", b);
  if (N == 0) return PW_OK;
  if (!planes || !idx) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  int rc = pw::check_device();
  if (rc) return rc;
  cudaError_t e = pw::launch_unpack_top(planes, N, K, b, idx, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "unpack launch");
}

int pw_route_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_ids,
                  float* topk_weights, cudaStream_t stream) {
  if (T < 0 || E <= 0 || k <= 0) return fail(PW_ERR_INVALID_ARG, "T < 0, E <= 0 or k <= 0");
  if (E > 1024 || k > 32 || k > E) return fail(PW_ERR_SHAPE, "limits: k <= min(E, 32), E <= 1024");
  if (T == 0) return PW_OK;
  if (!logits || !topk_ids || !topk_weights) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  int rc = pw::check_device();
  if (rc) return rc;
  cudaError_t e = pw::launch_route_topk(logits, T, E, k, topk_ids, topk_weights, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "route launch");
}

int pw_permute(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E, int32_t* offsets,
               int32_t* perm, int32_t* inv, int32_t* status_out, cudaStream_t stream) {
  if (T < 0 || k <= 0 || E <= 0) return fail(PW_ERR_INVALID_ARG, "T < 0, k <= 0 or E <= 0");
  if (E > 1024) return fail(PW_ERR_SHAPE, "E (%d) > 1024", E);
  if (static_cast<long long>(T) * k > (1LL << 30)) return fail(PW_ERR_SHAPE, "T*k too large");
  if (!offsets || (T > 0 && (!topk_ids || !perm)))
    return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  int rc = pw::check_device();
  if (rc) return rc;
  cudaError_t e = pw::launch_permute(topk_ids, T * k, E, offsets, perm, inv, status_out, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "permute launch");
}

int pw_page_table_create(int32_t num_blocks, const pw_block_entry* host_init,
                         pw_page_table** out) {
  if (out == nullptr) return fail(PW_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_blocks <= 0 || host_init == nullptr)
    return fail(PW_ERR_INVALID_ARG, "num_blocks must be > 0 and host_init non-NULL");
  for (int i = 0; i < num_blocks; ++i) {
    const pw_block_entry& b = host_init[i];
    if (!pw::supported_q_host(b.q))
      return fail(PW_ERR_UNSUPPORTED_Q, "block %d: q = %d is not in {3,4,5,6,8}", i, b.q);
    if (b.state < PW_PAGE_GPU || b.state > PW_PAGE_IN_TRANSFER)
      return fail(PW_ERR_INVALID_ARG, "block %d: page state %d unknown", i, b.state);
    if (!b.planes || !b.lut || !pw::aligned(b.planes, 16) || !pw::aligned(b.lut, 16))
      return fail(PW_ERR_INVALID_ARG, "block %d: planes/lut NULL or not 16-byte aligned", i);
  }
  int rc = pw::check_device();
  if (rc) return rc;
  pw_page_table* t = new (std::nothrow) pw_page_table();
  if (!t) return fail(PW_ERR_INVALID_ARG, "out of host memory");
  cudaError_t e = cudaGetDevice(&t->device);
  if (e == cudaSuccess) e = cudaMalloc(&t->d_entries, sizeof(pw_block_entry) * num_blocks);
  if (e == cudaSuccess) e = cudaMalloc(&t->d_status, sizeof(int32_t));
  if (e == cudaSuccess)
    e = cudaMemcpy(t->d_entries, host_init, sizeof(pw_block_entry) * num_blocks,
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(t->d_status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(t->d_entries);
    cudaFree(t->d_status);
    delete t;
    return cuda_fail(e, "page table create");
  }
  t->num_blocks = num_blocks;
  *out = t;
  return PW_OK;
}

int pw_page_table_set_routing_stats(pw_page_table* t, int32_t* counts, float* mass) {
  if (t == nullptr) return fail(PW_ERR_INVALID_ARG, "table is NULL");
  if ((counts == nullptr) != (mass == nullptr))
    return fail(PW_ERR_INVALID_ARG, "pass both statistics buffers or neither");
  t->stats_counts = counts;
  t->stats_mass = mass;
  return PW_OK;
}

int pw_page_table_destroy(pw_page_table* t) {
  if (t == nullptr) return PW_OK;
  cudaError_t e = cudaDeviceSynchronize();
  cudaFree(t->d_entries);
  cudaFree(t->d_status);
  delete t;
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "page table destroy");
}

int pw_page_table_commit(pw_page_table* t, int32_t n, const int32_t* block_ids,
                         const int32_t* new_q, const uint16_t* const* new_lut,
                         cudaStream_t stream) {
  return pw::update_table(t, n, block_ids, 0, new_q, reinterpret_cast<const void* const*>(new_lut),
                          stream);
}

int pw_page_table_set_pages(pw_page_table* t, int32_t n, const int32_t* block_ids,
                            const uint32_t* const* planes, const int32_t* states,
                            cudaStream_t stream) {
  return pw::update_table(t, n, block_ids, 1, states, reinterpret_cast<const void* const*>(planes),
                          stream);
}

int pw_page_table_commit_after(pw_page_table* t, int32_t n, const int32_t* block_ids,
                               const int32_t* new_q, const uint16_t* const* new_lut,
                               cudaEvent_t ready, cudaStream_t stream) {
  if (ready != nullptr) {
    cudaError_t e = cudaStreamWaitEvent(stream, ready, 0);
    if (e != cudaSuccess) return cuda_fail(e, "wait for the page copy");
  }
  return pw_page_table_commit(t, n, block_ids, new_q, new_lut, stream);
}

namespace pw {
namespace {

int plane_tail_args(const void* dev, const void* host, int32_t N, int32_t K, int32_t p_begin,
                    size_t* bytes, size_t* offset) {
  if (N < 0) return fail(PW_ERR_INVALID_ARG, "N < 0");
  if (K <= 0 || K % 32) return fail(PW_ERR_SHAPE, "K (%d) must be a positive multiple of 32", K);
  if (p_begin < 0 || p_begin > 7) return fail(PW_ERR_INVALID_ARG, "p_begin %d outside 0..7", p_begin);
  if (!dev || !host || !aligned(dev, 16))
    return fail(PW_ERR_INVALID_ARG, "NULL pointer or planes not 16-byte aligned");
  const size_t plane = static_cast<size_t>(N) * (K / 32) * 4;
  *bytes = plane * static_cast<size_t>(8 - p_begin);
  *offset = plane * static_cast<size_t>(p_begin);
  return PW_OK;
}

}  // namespace
}  // namespace pw

int pw_planes_to_host(const uint32_t* planes, int32_t N, int32_t K, int32_t p_begin, void* host,
                      cudaStream_t stream) {
  size_t bytes = 0, off = 0;
  int rc = pw::plane_tail_args(planes, host, N, K, p_begin, &bytes, &off);
  if (rc) return rc;
  if (bytes == 0) return PW_OK;
  cudaError_t e = cudaMemcpyAsync(host, reinterpret_cast<const char*>(planes) + off, bytes,
                                  cudaMemcpyDeviceToHost, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "planes to host");
}

int pw_planes_from_host(const void* host, uint32_t* planes, int32_t N, int32_t K, int32_t p_begin,
                        cudaStream_t stream) {
  size_t bytes = 0, off = 0;
  int rc = pw::plane_tail_args(planes, host, N, K, p_begin, &bytes, &off);
  if (rc) return rc;
  if (bytes == 0) return PW_OK;
  cudaError_t e = cudaMemcpyAsync(reinterpret_cast<char*>(planes) + off, host, bytes,
                                  cudaMemcpyHostToDevice, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "planes from host");
}

int pw_page_table_read(const pw_page_table* t, pw_block_entry* host_out, cudaStream_t stream) {
  if (!t || !host_out) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = cudaMemcpyAsync(host_out, t->d_entries, sizeof(pw_block_entry) * t->num_blocks,
                                  cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "page table read");
}

int32_t pw_page_table_size(const pw_page_table* t) { return t ? t->num_blocks : 0; }

int pw_page_table_status(pw_page_table* t, int32_t* host_status, int32_t reset,
                         cudaStream_t stream) {
  if (!t || !host_status) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = cudaMemcpyAsync(host_status, t->d_status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  stream);
  if (e == cudaSuccess && reset) e = cudaMemsetAsync(t->d_status, 0, sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "page table status");
}

int pw_workspace_bytes(const pw_moe_shape* shape, size_t* bytes) {
  if (!bytes) return fail(PW_ERR_INVALID_ARG, "bytes is NULL");
  int rc = pw::check_shape(shape);
  if (rc) return rc;
  const size_t d = pw::decode_workspace_bytes(*shape);
  const size_t p = pw::prefill_workspace_bytes(*shape);
  *bytes = d > p ? d : p;
  return PW_OK;
}

int pw_moe_forward(const pw_moe_shape* shape, const void* hidden, const int32_t* topk_ids,
                   const float* topk_weights, const pw_page_table* table, float* out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return pw::forward_impl(shape, hidden, topk_ids, topk_weights, table, out, workspace,
                          workspace_bytes, PW_PATH_AUTO, stream);
}

int pw_moe_forward_path(const pw_moe_shape* shape, const void* hidden, const int32_t* topk_ids,
                        const float* topk_weights, const pw_page_table* table, float* out,
                        void* workspace, size_t workspace_bytes, int32_t path,
                        cudaStream_t stream) {
  return pw::forward_impl(shape, hidden, topk_ids, topk_weights, table, out, workspace,
                          workspace_bytes, path, stream);
}

int pw_debug_bounded_wait(pw_page_table* table, int32_t which, int32_t polls,
                          cudaStream_t stream) {
  if (table == nullptr) return fail(PW_ERR_INVALID_ARG, "table is NULL");
  if (which != 0 && which != 1) return fail(PW_ERR_INVALID_ARG, "which must be 0 or 1");
  if (polls < 1 || polls > (1 << 20)) return fail(PW_ERR_INVALID_ARG, "polls outside 1..2^20");
  int rc = pw::check_device();
  if (rc) return rc;
  const cudaError_t e =
      which == 0 ? pw::launch_wait_check_decode(table->d_status, static_cast<uint32_t>(polls), stream)
                 : pw::launch_wait_check_mbar(table->d_status, static_cast<uint32_t>(polls), stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "bounded-wait check launch");
}

int pw_debug_gemm_trace(void* host, size_t bytes, size_t* needed) {
  if (needed) *needed = pw::gemm_trace_bytes();
  if (host == nullptr || bytes < pw::gemm_trace_bytes())
    return fail(PW_ERR_INVALID_ARG, "host buffer NULL or smaller than %zu bytes",
                pw::gemm_trace_bytes());
  int rc = pw::check_device();
  if (rc) return rc;
  cudaError_t e = cudaSuccess;
  if (!pw::gemm_trace_read(host, bytes, &e))
    return fail(PW_ERR_NOT_BUILT, "libpw was built without the GEMM trace (build.py --trace)");
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "trace copy");
}

int pw_debug_decode_trace(void* host, size_t bytes, size_t* needed) {
  if (needed) *needed = pw::decode_trace_bytes();
  if (host == nullptr || bytes < pw::decode_trace_bytes())
    return fail(PW_ERR_INVALID_ARG, "host buffer NULL or smaller than %zu bytes",
                pw::decode_trace_bytes());
  int rc = pw::check_device();
  if (rc) return rc;
  cudaError_t e = cudaSuccess;
  if (!pw::decode_trace_read(host, bytes, &e))
    return fail(PW_ERR_NOT_BUILT, "libpw was built without the decode trace (build.py --trace)");
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "trace copy");
}

int pw_debug_index(const uint32_t* planes, int32_t N, int32_t K, int32_t q, int32_t form,
                   uint8_t* idx, cudaStream_t stream) {
  if (N < 0) return fail(PW_ERR_INVALID_ARG, "N < 0");
  if (K <= 0 || K % 32) return fail(PW_ERR_SHAPE, "K (%d) must be a positive multiple of 32", K);
  if (!pw::supported_q_host(q)) return fail(PW_ERR_UNSUPPORTED_Q, "q = %d is not in {3,4,5,6,8}", q);
  if (form < PW_INDEX_NIBBLES || form > PW_INDEX_HALVES)
    return fail(PW_ERR_INVALID_ARG, "unknown index form %d", form);
  if (form == PW_INDEX_NIBBLES && q > 4)
    return fail(PW_ERR_UNSUPPORTED_Q, "nibble indices hold q <= 4 (got %d)", q);
  if (N == 0) return PW_OK;
  if (!planes || !idx) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  int rc = pw::check_device();
  if (rc) return rc;
  const cudaError_t e =
      form == PW_INDEX_HALVES ? pw::launch_half_index_check(planes, N, K, q, idx, stream)
                              : pw::launch_index_check(planes, N, K, q, form == PW_INDEX_NIBBLES, idx, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "index check launch");
}

int pw_debug_dequant(const uint32_t* planes, const uint16_t* lut, int32_t N, int32_t K, int32_t q,
                     int32_t path, float* w, pw_page_table* table, cudaStream_t stream) {
  if (N < 0) return fail(PW_ERR_INVALID_ARG, "N < 0");
  if (K <= 0 || K % 32) return fail(PW_ERR_SHAPE, "K (%d) must be a positive multiple of 32", K);
  if (N % 32) return fail(PW_ERR_SHAPE, "N (%d) must be a multiple of 32", N);
  if (!pw::supported_q_host(q)) return fail(PW_ERR_UNSUPPORTED_Q, "q = %d is not in {3,4,5,6,8}", q);
  if (path != PW_PATH_DECODE && path != PW_PATH_PREFILL)
    return fail(PW_ERR_INVALID_ARG, "path must be PW_PATH_DECODE or PW_PATH_PREFILL");
  if (N == 0) return PW_OK;
  if (!planes || !lut || !w) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  if (!pw::aligned(lut, 16)) return fail(PW_ERR_INVALID_ARG, "lut must be 16-byte aligned");
  int rc = pw::check_device();
  if (rc) return rc;
  const cudaError_t e =
      path == PW_PATH_PREFILL
          ? pw::launch_half_dequant_check(planes, lut, N, K, q, w, stream)
          : pw::launch_dequant_check(planes, lut, N, K, q, w, table ? table->d_status : nullptr, stream);
  return e == cudaSuccess ? PW_OK : cuda_fail(e, "dequant check launch");
}

int pw_debug_workspace_section(const pw_moe_shape* shape, int32_t path, int32_t section,
                               size_t* offset, size_t* bytes) {
  int rc = pw::check_shape(shape);
  if (rc) return rc;
  if (!offset || !bytes) return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  if (path != PW_PATH_DECODE && path != PW_PATH_PREFILL)
    return fail(PW_ERR_INVALID_ARG, "path must be PW_PATH_DECODE or PW_PATH_PREFILL");
  const int r = path == PW_PATH_DECODE ? pw::decode_ws_section(*shape, section, offset, bytes)
                                       : pw::prefill_ws_section(*shape, section, offset, bytes);
  return r == 0 ? PW_OK : fail(PW_ERR_INVALID_ARG, "unknown workspace section %d", section);
}

int pw_moe_forward_logits(const pw_moe_shape* shape, const void* hidden, const float* logits,
                          int32_t* topk_ids, float* topk_weights, const pw_page_table* table,
                          float* out, void* workspace, size_t workspace_bytes, int32_t path,
                          cudaStream_t stream) {
  if (logits == nullptr && shape != nullptr && shape->T > 0)
    return fail(PW_ERR_INVALID_ARG, "logits is NULL");
  return pw::forward_impl(shape, hidden, topk_ids, topk_weights, table, out, workspace,
                          workspace_bytes, path, stream, logits);
}

int32_t pw_prefill_min_pairs(const pw_moe_shape* shape) {
  if (pw::check_shape(shape)) return -1;
  return pw::prefill_min_pairs(*shape);
}

}  // extern "C"
