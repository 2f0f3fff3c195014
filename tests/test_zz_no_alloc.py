"""pw_moe_forward_noalloc against pw_moe_forward, through the C ABI.

pw_moe_forward_noalloc serves callers that have no way to get device memory
for a workspace (plugin hooks that are only handed their inputs and outputs,
runtimes that fix their memory budget at start-up, code where an allocation
would synchronise the device).  It runs the same decode kernels with their
scratch in a fixed static device array inside the library.  This file sits
last in collection order so that a stop-at-first-failure run has already run
every other test; it also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from helpers import REL_TOL, host_layer, oracle_route, rel_l2
from workloads import gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pw():
    import any_precision_bitplane_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.lib()
    return m


def _noalloc(pw, shape, hidden, ids, w, table, out):
    rc = pw.lib().pw_moe_forward_noalloc(ctypes.byref(shape), ctypes.c_void_p(hidden.data_ptr()),
                                         ctypes.c_void_p(ids.data_ptr()),
                                         ctypes.c_void_p(w.data_ptr()), table.handle,
                                         ctypes.c_void_p(out.data_ptr()),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("name,T", [("tiny", 16), ("qwen3_decode", 64)])
def test_noalloc_matches_forward_twice(pw, name, T):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = host_layer(name)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids_np, w_np = oracle_route(tok, layer.cfg.k)
        hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
        ids = torch.from_numpy(ids_np).cuda()
        w = torch.from_numpy(w_np).cuda()
        ref = pw.moe_forward(hidden, ids, w, dl.table, dl.I, dl.E).cpu().numpy()
        shape = pw.MoeShape(T, dl.H, dl.I, dl.E, layer.cfg.k)
        for _ in range(2):   # two calls in a row share (and reuse) the static scratch
            out = torch.full((T, dl.H), float("nan"), dtype=torch.float32, device="cuda")
            rc = _noalloc(pw, shape, hidden, ids, w, dl.table, out)
            assert rc == pw.PW_OK, pw.last_error()
            got = out.cpu().numpy()
            assert np.isfinite(got).all()
            assert rel_l2(got, ref) <= REL_TOL
        assert dl.table.status() == pw.PW_OK
    finally:
        dl.close()


def test_noalloc_rejects_shapes_beyond_its_scratch(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = host_layer("tiny")
    dl = DeviceLayer(layer)
    try:
        T = 2048   # 2048 tokens x top-2 x (512 + 256) x 4 bytes = 12 MiB > 8 MiB
        hidden = torch.zeros((T, dl.H), dtype=torch.int16, device="cuda")
        ids = torch.zeros((T, 2), dtype=torch.int32, device="cuda")
        w = torch.zeros((T, 2), dtype=torch.float32, device="cuda")
        out = torch.zeros((T, dl.H), dtype=torch.float32, device="cuda")
        rc = _noalloc(pw, pw.MoeShape(T, dl.H, dl.I, dl.E, 2), hidden, ids, w, dl.table, out)
        assert rc == pw.PW_ERR_WORKSPACE
        assert "static scratch" in pw.last_error()
    finally:
        dl.close()


def test_noalloc_from_two_host_threads(pw):
    # the library's host state (the cached scratch address, per-device set-up)
    # is shared by threads; two threads enqueue no-alloc calls onto one
    # stream (the documented ordering for the shared scratch), each with its
    # own tokens, and every result matches the workspace path
    import threading
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = host_layer("tiny")
    dl = DeviceLayer(layer)
    try:
        stream = torch.cuda.current_stream()
        jobs = []
        for seed_T in (16, 12):
            tok = gen.make_tokens(layer, seed_T)
            ids_np, w_np = oracle_route(tok, layer.cfg.k)
            hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
            ids = torch.from_numpy(ids_np).cuda()
            w = torch.from_numpy(w_np).cuda()
            ref = pw.moe_forward(hidden, ids, w, dl.table, dl.I, dl.E).cpu().numpy()
            outs = [torch.full((seed_T, dl.H), float("nan"), dtype=torch.float32, device="cuda")
                    for _ in range(3)]
            jobs.append((pw.MoeShape(seed_T, dl.H, dl.I, dl.E, layer.cfg.k), hidden, ids, w, ref,
                         outs))
        torch.cuda.synchronize()
        codes = []

        def run(job):
            shape, hidden, ids, w, _, outs = job
            for out in outs:
                rc = pw.lib().pw_moe_forward_noalloc(
                    ctypes.byref(shape), ctypes.c_void_p(hidden.data_ptr()),
                    ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                    dl.table.handle, ctypes.c_void_p(out.data_ptr()),
                    ctypes.c_void_p(stream.cuda_stream))
                codes.append(rc)

        threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        torch.cuda.synchronize()
        assert codes == [pw.PW_OK] * 6
        for _, _, _, _, ref, outs in jobs:
            for out in outs:
                assert rel_l2(out.cpu().numpy(), ref) <= REL_TOL
        assert dl.table.status() == pw.PW_OK
    finally:
        dl.close()
