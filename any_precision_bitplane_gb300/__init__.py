"""PagedWeight fused mixed-precision MoE layer on GB300 (sm_103a).

Python binding of libpw.so.  Every function here only marshals arguments
(torch tensors -> device pointers, the current CUDA stream) and calls the C
ABI declared in include/pw.h; all computation runs in the library's CUDA
kernels.  There is no fallback: if libpw.so is missing or cannot load, every
call raises.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpw.so")

PW_OK = 0
PW_ERR_INVALID_ARG = 1
PW_ERR_UNSUPPORTED_Q = 2
PW_ERR_SHAPE = 3
PW_ERR_WORKSPACE = 4
PW_ERR_PAGE_NOT_RESIDENT = 5
PW_ERR_BAD_EXPERT_ID = 6
PW_ERR_CUDA = 7
PW_ERR_TIMEOUT = 8
PW_ERR_UNSUPPORTED_DEVICE = 9
PW_ERR_RANGE = 10
PW_ERR_NOT_BUILT = 11

PW_PAGE_GPU = 0
PW_PAGE_CPU = 1
PW_PAGE_IN_TRANSFER = 2

PATH_AUTO = 0
PATH_DECODE = 1
PATH_PREFILL = 2

INDEX_NIBBLES = 0
INDEX_BYTES = 1
INDEX_HALVES = 2

BITWIDTHS = (3, 4, 5, 6, 8)


class PWError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(msg)
        self.code = code


class BlockEntry(ctypes.Structure):
    _fields_ = [("q", ctypes.c_int32), ("state", ctypes.c_int32),
                ("planes", ctypes.c_void_p), ("lut", ctypes.c_void_p)]


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


_c = ctypes
_P = _c.c_void_p
_I32 = _c.c_int32
_SIGNATURES = {
    "pw_last_error": (_c.c_char_p, []),
    "pw_version": (_c.c_int, []),
    "pw_pack_bitplanes": (_c.c_int, [_P, _I32, _I32, _P, _P]),
    "pw_unpack_top": (_c.c_int, [_P, _I32, _I32, _I32, _P, _P]),
    "pw_route_topk": (_c.c_int, [_P, _I32, _I32, _I32, _P, _P, _P]),
    "pw_permute": (_c.c_int, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "pw_page_table_create": (_c.c_int, [_I32, _P, _P]),
    "pw_page_table_destroy": (_c.c_int, [_P]),
    "pw_page_table_commit": (_c.c_int, [_P, _I32, _P, _P, _P, _P]),
    "pw_page_table_set_pages": (_c.c_int, [_P, _I32, _P, _P, _P, _P]),
    "pw_page_table_read": (_c.c_int, [_P, _P, _P]),
    "pw_page_table_size": (_I32, [_P]),
    "pw_page_table_status": (_c.c_int, [_P, _P, _I32, _P]),
    "pw_workspace_bytes": (_c.c_int, [_P, _P]),
    "pw_moe_forward": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P, _c.c_size_t, _P]),
    "pw_moe_forward_path": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P, _c.c_size_t, _I32, _P]),
    "pw_prefill_min_pairs": (_I32, [_P]),
    "pw_moe_forward_noalloc": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    "pw_set_timing_events": (_c.c_int, [_P, _P]),
    "pw_page_table_set_routing_stats": (_c.c_int, [_P, _P, _P]),
    "pw_planes_to_host": (_c.c_int, [_P, _I32, _I32, _I32, _P, _P]),
    "pw_planes_from_host": (_c.c_int, [_P, _P, _I32, _I32, _I32, _P]),
    "pw_page_table_commit_after": (_c.c_int, [_P, _I32, _P, _P, _P, _P, _P]),
    "pw_plan_recommit": (_c.c_int, [_I32, _P, _P, _P, _P, _I32, _c.c_int64, _P, _P, _P, _P]),
    "pw_debug_bounded_wait": (_c.c_int, [_P, _I32, _I32, _P]),
    "pw_debug_gemm_trace": (_c.c_int, [_P, _c.c_size_t, _P]),
    "pw_debug_decode_trace": (_c.c_int, [_P, _c.c_size_t, _P]),
    "pw_debug_index": (_c.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P]),
    "pw_debug_dequant": (_c.c_int, [_P, _P, _I32, _I32, _I32, _I32, _P, _P, _P]),
    "pw_debug_workspace_section": (_c.c_int, [_P, _I32, _I32, _P, _P]),
    "pw_moe_forward_logits": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _c.c_size_t, _I32, _P]),
}
EXPORTED = tuple(_SIGNATURES)

_lib = None


def lib():
    """The loaded libpw.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise PWError(PW_ERR_INVALID_ARG,
                          "libpw.so not built (expected at %s); run "
                          "python any_precision_bitplane_gb300/build.py" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def last_error():
    return lib().pw_last_error().decode()


def _check(rc, name):
    if rc != PW_OK:
        raise PWError(rc, "%s failed (status %d): %s" % (name, rc, last_error()))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise PWError(PW_ERR_INVALID_ARG, "tensors must be contiguous CUDA tensors")


# ---------------------------------------------------------------- bitplanes

def pack_bitplanes(codes, planes=None, stream=None):
    """codes uint8 [N, K] -> planes int32 [8, K/32, N] (raw uint32 bits)."""
    _need_cuda(codes)
    N, K = codes.shape
    if planes is None:
        planes = torch.empty((8, K // 32, N), dtype=torch.int32, device=codes.device)
    _need_cuda(planes)
    _check(lib().pw_pack_bitplanes(_ptr(codes), N, K, _ptr(planes), _stream(stream)),
           "pw_pack_bitplanes")
    return planes


def unpack_top(planes, N, K, b, idx=None, stream=None):
    """Top-b planes -> uint8 indices [N, K] (= code >> (8-b))."""
    _need_cuda(planes)
    if idx is None:
        idx = torch.empty((N, K), dtype=torch.uint8, device=planes.device)
    _check(lib().pw_unpack_top(_ptr(planes), N, K, b, _ptr(idx), _stream(stream)),
           "pw_unpack_top")
    return idx


# ---------------------------------------------------------------- routing

def route_topk(logits, k, ids=None, weights=None, stream=None):
    """float32 logits [T, E] -> (int32 ids [T, k], float32 weights [T, k])."""
    _need_cuda(logits)
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().pw_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(weights), _stream(stream)),
           "pw_route_topk")
    return ids, weights


def permute(topk_ids, E, with_inv=True, status=None, stream=None):
    """int32 ids [T, k] -> (offsets [E+1], perm [T*k], inv [T*k] or None)."""
    _need_cuda(topk_ids)
    T, k = topk_ids.shape
    dev = topk_ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)[:T * k]
    inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)[:T * k] if with_inv else None
    _check(lib().pw_permute(_ptr(topk_ids), T, k, E, _ptr(offsets), _ptr(perm), _ptr(inv),
                            _ptr(status), _stream(stream)), "pw_permute")
    return offsets, perm, inv


# ---------------------------------------------------------------- page table

class PageTable:
    """Weight Page Table: per block (q, state, planes pointer, LUT pointer).

    The table's device array never moves, so forward calls captured in a CUDA
    graph read whatever was committed last on the stream.
    """

    def __init__(self, entries):
        arr = (BlockEntry * len(entries))()
        for i, (q, state, planes_ptr, lut_ptr) in enumerate(entries):
            arr[i] = BlockEntry(int(q), int(state), int(planes_ptr), int(lut_ptr))
        handle = ctypes.c_void_p()
        _check(lib().pw_page_table_create(len(entries), arr, ctypes.byref(handle)),
               "pw_page_table_create")
        self.handle = handle
        self.num_blocks = len(entries)

    def commit(self, block_ids, new_q, new_lut_ptrs, stream=None):
        n = len(block_ids)
        ids = (ctypes.c_int32 * max(n, 1))(*[int(b) for b in block_ids])
        qs = (ctypes.c_int32 * max(n, 1))(*[int(q) for q in new_q])
        luts = (ctypes.c_void_p * max(n, 1))(*[int(p) for p in new_lut_ptrs])
        _check(lib().pw_page_table_commit(self.handle, n, ids, qs, luts, _stream(stream)),
               "pw_page_table_commit")

    def commit_after(self, block_ids, new_q, new_lut_ptrs, ready, stream=None):
        """commit() ordered after torch.cuda.Event `ready` (e.g. a page reload)."""
        n = len(block_ids)
        ids = (ctypes.c_int32 * max(n, 1))(*[int(b) for b in block_ids])
        qs = (ctypes.c_int32 * max(n, 1))(*[int(q) for q in new_q])
        luts = (ctypes.c_void_p * max(n, 1))(*[int(p) for p in new_lut_ptrs])
        _check(lib().pw_page_table_commit_after(self.handle, n, ids, qs, luts,
                                                ctypes.c_void_p(ready.cuda_event), _stream(stream)),
               "pw_page_table_commit_after")

    def set_pages(self, block_ids, planes_ptrs, states, stream=None):
        n = len(block_ids)
        ids = (ctypes.c_int32 * max(n, 1))(*[int(b) for b in block_ids])
        pl = (ctypes.c_void_p * max(n, 1))(*[int(p) for p in planes_ptrs])
        st = (ctypes.c_int32 * max(n, 1))(*[int(s) for s in states])
        _check(lib().pw_page_table_set_pages(self.handle, n, ids, pl, st, _stream(stream)),
               "pw_page_table_set_pages")

    def read(self, stream=None):
        arr = (BlockEntry * self.num_blocks)()
        _check(lib().pw_page_table_read(self.handle, arr, _stream(stream)), "pw_page_table_read")
        return [(e.q, e.state, e.planes or 0, e.lut or 0) for e in arr]

    def status(self, reset=True, stream=None):
        v = ctypes.c_int32(0)
        _check(lib().pw_page_table_status(self.handle, ctypes.byref(v), 1 if reset else 0,
                                          _stream(stream)), "pw_page_table_status")
        return v.value

    def set_routing_stats(self, counts=None, mass=None):
        """Accumulate per-expert routing statistics into `counts` (int32 [E]) and
        `mass` (float32 [E]) during every following forward call; None stops."""
        if counts is not None:
            _need_cuda(counts, mass)
        self._stats = (counts, mass)   # keep the buffers alive while attached
        _check(lib().pw_page_table_set_routing_stats(
            self.handle, _ptr(counts) if counts is not None else None,
            _ptr(mass) if mass is not None else None), "pw_page_table_set_routing_stats")

    def close(self):
        if self.handle is not None and self.handle.value:
            _check(lib().pw_page_table_destroy(self.handle), "pw_page_table_destroy")
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- the layer

def shape(T, H, I, E, k):
    return MoeShape(T, H, I, E, k)


def workspace_bytes(T, H, I, E, k):
    n = ctypes.c_size_t(0)
    s = MoeShape(T, H, I, E, k)
    _check(lib().pw_workspace_bytes(ctypes.byref(s), ctypes.byref(n)), "pw_workspace_bytes")
    return n.value


def prefill_min_pairs(T, H, I, E, k):
    s = MoeShape(T, H, I, E, k)
    return int(lib().pw_prefill_min_pairs(ctypes.byref(s)))


def moe_forward(hidden, topk_ids, topk_weights, table, I, E, out=None, workspace=None,
                path=PATH_AUTO, stream=None):
    """out[t] = sum_j w_tj * expert_{e_tj}(hidden[t]) with every block at its committed q.

    hidden: bf16 [T, H] (torch.bfloat16 or raw int16 bits), topk_ids int32 [T, k],
    topk_weights float32 [T, k], table: PageTable with 2E blocks.
    """
    _need_cuda(hidden, topk_ids, topk_weights)
    T, H = hidden.shape
    k = topk_ids.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=hidden.device)
    _need_cuda(out)
    need = workspace_bytes(T, H, I, E, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=hidden.device)
    _need_cuda(workspace)
    s = MoeShape(T, H, I, E, k)
    _check(lib().pw_moe_forward_path(ctypes.byref(s), _ptr(hidden), _ptr(topk_ids),
                                     _ptr(topk_weights), table.handle, _ptr(out),
                                     _ptr(workspace), workspace.numel(), int(path),
                                     _stream(stream)), "pw_moe_forward")
    return out


def moe_forward_logits(hidden, logits, table, I, E, k, out=None, workspace=None, ids=None,
                       weights=None, path=PATH_AUTO, stream=None):
    """The layer fed with router logits [T, E] (float32): the routing runs
    inside the call.  Returns (out, topk ids int32 [T, k], topk weights
    float32 [T, k])."""
    _need_cuda(hidden, logits)
    T, H = hidden.shape
    dev = hidden.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=dev)
    _need_cuda(out, ids, weights)
    need = workspace_bytes(T, H, I, E, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    s = MoeShape(T, H, I, E, k)
    _check(lib().pw_moe_forward_logits(ctypes.byref(s), _ptr(hidden), _ptr(logits), _ptr(ids),
                                       _ptr(weights), table.handle, _ptr(out), _ptr(workspace),
                                       workspace.numel(), int(path), _stream(stream)),
           "pw_moe_forward_logits")
    return out, ids, weights


def moe_forward_noalloc(hidden, topk_ids, topk_weights, table, I, E, out=None, stream=None):
    """moe_forward without a workspace: the library's fixed static scratch is
    used instead (decode path; shapes whose scratch exceeds it raise)."""
    _need_cuda(hidden, topk_ids, topk_weights)
    T, H = hidden.shape
    k = topk_ids.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=hidden.device)
    _need_cuda(out)
    s = MoeShape(T, H, I, E, k)
    _check(lib().pw_moe_forward_noalloc(ctypes.byref(s), _ptr(hidden), _ptr(topk_ids),
                                        _ptr(topk_weights), table.handle, _ptr(out),
                                        _stream(stream)), "pw_moe_forward_noalloc")
    return out


def debug_bounded_wait(table, which, polls, stream=None):
    """Run one of the forward kernels' bounded device waits (0: the decode
    down kernel's wait for gate_up tiles, 1: the tensor-core kernels'
    mbarrier wait) against something never released, with `polls` as its
    limit; it latches PW_ERR_TIMEOUT in the table's status word."""
    _check(lib().pw_debug_bounded_wait(table.handle, int(which), int(polls), _stream(stream)),
           "pw_debug_bounded_wait")


TRACE_LIB_PATH = os.path.join(_PKG, "libpw_trace.so")


def debug_gemm_trace():
    """The gate_up GEMM's pipeline trace of the last launch (a library built
    with build.py --trace): (step uint64 [16, 256, 4], tile uint64 [16, 32, 6],
    smid uint64 [16], dq uint64 [16, 256, 8, 4]) for CTAs 0, 10, ..., 150;
    %globaltimer nanoseconds, 0 where not reached; smid is the SM id plus one.  Raises PWError
    (PW_ERR_NOT_BUILT) on a library built without tracing."""
    import numpy as np
    need = ctypes.c_size_t(0)
    lib().pw_debug_gemm_trace(None, 0, ctypes.byref(need))
    buf = np.zeros(need.value // 8, dtype=np.uint64)
    _check(lib().pw_debug_gemm_trace(buf.ctypes.data, buf.nbytes, None), "pw_debug_gemm_trace")
    n_step, n_dq, n_tile = 16 * 256 * 4, 16 * 256 * 8 * 4, 16 * 32 * 6
    step = buf[:n_step].reshape(16, 256, 4)
    dq = buf[n_step:n_step + n_dq].reshape(16, 256, 8, 4)
    tile = buf[n_step + n_dq:n_step + n_dq + n_tile].reshape(16, 32, 6)
    smid = buf[n_step + n_dq + n_tile:n_step + n_dq + n_tile + 16]
    return step, tile, smid, dq


def debug_decode_trace():
    """The decode gate_up kernel's per-tile phase trace of the last launch (a
    library built with build.py --trace): (tile uint64 [16, 32, 10], cta uint64
    [16, 2]) for CTAs 0, 19, ..., 285; tile fields: start ns, end ns, then SM
    cycles of descriptor, set-up, columns, reduction + store, then q + 256 *
    pairs, then the set-up's parts (issue, LUT wait + build, barrier); cta: SM
    id + 1, exit ns.  Raises PWError (PW_ERR_NOT_BUILT) on a
    library built without tracing."""
    import numpy as np
    need = ctypes.c_size_t(0)
    lib().pw_debug_decode_trace(None, 0, ctypes.byref(need))
    buf = np.zeros(need.value // 8, dtype=np.uint64)
    _check(lib().pw_debug_decode_trace(buf.ctypes.data, buf.nbytes, None),
           "pw_debug_decode_trace")
    n_tile = 16 * 32 * 10
    return buf[:n_tile].reshape(16, 32, 10), buf[n_tile:n_tile + 32].reshape(16, 2)


def debug_index(planes, N, K, q, form, idx=None, stream=None):
    """The kernels' own index extraction (form INDEX_NIBBLES / INDEX_BYTES /
    INDEX_HALVES) on a block: uint8 [N, K], column order restored."""
    _need_cuda(planes)
    if idx is None:
        idx = torch.empty((N, K), dtype=torch.uint8, device=planes.device)
    _check(lib().pw_debug_index(_ptr(planes), N, K, q, form, _ptr(idx), _stream(stream)),
           "pw_debug_index")
    return idx


def debug_dequant(planes, lut, N, K, q, path, table=None, out=None, stream=None):
    """The kernels' own table build and lookup on a block (path PATH_DECODE or
    PATH_PREFILL): float32 [N, K]."""
    _need_cuda(planes, lut)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=planes.device)
    _check(lib().pw_debug_dequant(_ptr(planes), _ptr(lut), N, K, q, path, _ptr(out),
                                  table.handle if table is not None else None, _stream(stream)),
           "pw_debug_dequant")
    return out


def debug_workspace_section(T, H, I, E, k, path, section):
    """(offset, bytes) of a section of a forward call's workspace."""
    s = MoeShape(T, H, I, E, k)
    off = ctypes.c_size_t(0)
    n = ctypes.c_size_t(0)
    _check(lib().pw_debug_workspace_section(ctypes.byref(s), path, section, ctypes.byref(off),
                                            ctypes.byref(n)), "pw_debug_workspace_section")
    return off.value, n.value


def set_timing_events(before=None, after=None):
    """Record torch.cuda.Event `before` / `after` (timing enabled, already
    recorded once so that they exist) around the dominant kernel of every
    following forward call; None, None stops."""
    b = before.cuda_event if before is not None else None
    a = after.cuda_event if after is not None else None
    _check(lib().pw_set_timing_events(b, a), "pw_set_timing_events")


def plan_recommit(q_now, sensitivity, bytes_per_bit, routing_mass, hot_floor, bytes_to_free):
    """Greedy damage-per-byte planner (host computation in libpw).  Arrays are
    host sequences of length 2E (routing_mass: E).  Returns (block ids,
    new bitwidths, bytes freed): the list a PageTable.commit applies."""
    import numpy as np
    q = np.ascontiguousarray(q_now, dtype=np.int32)
    s = np.ascontiguousarray(sensitivity, dtype=np.float32)
    b = np.ascontiguousarray(bytes_per_bit, dtype=np.int64)
    m = np.ascontiguousarray(routing_mass, dtype=np.float32)
    n = q.size
    ids = np.zeros(max(n, 1), dtype=np.int32)
    qs = np.zeros(max(n, 1), dtype=np.int32)
    n_out = ctypes.c_int32(0)
    freed = ctypes.c_int64(0)
    _check(lib().pw_plan_recommit(n, q.ctypes.data, s.ctypes.data, b.ctypes.data, m.ctypes.data,
                                  int(hot_floor), int(bytes_to_free), ids.ctypes.data,
                                  qs.ctypes.data, ctypes.byref(n_out), ctypes.byref(freed)),
           "pw_plan_recommit")
    k = n_out.value
    return ids[:k].tolist(), qs[:k].tolist(), freed.value


def planes_to_host(planes, N, K, p_begin, host, stream=None):
    """Copy planes [p_begin, 8) of a block (device tensor viewed as uint32
    [8][K/32][N]) into `host` (pinned CPU tensor of (8-p_begin)*N*K/8 bytes),
    asynchronously on `stream`."""
    _need_cuda(planes)
    _check(lib().pw_planes_to_host(_ptr(planes), N, K, p_begin, ctypes.c_void_p(host.data_ptr()),
                                   _stream(stream)), "pw_planes_to_host")


def planes_from_host(host, planes, N, K, p_begin, stream=None):
    """Copy `host` back into planes [p_begin, 8) of a block, asynchronously."""
    _need_cuda(planes)
    _check(lib().pw_planes_from_host(ctypes.c_void_p(host.data_ptr()), _ptr(planes), N, K, p_begin,
                                     _stream(stream)), "pw_planes_from_host")
