"""pw_moe_forward with pinned host buffers for hidden, topk ids, topk weights
and out (the kernels read and write them directly): bit-identical to the same
call on device buffers, on the decode and the prefill path."""
import ctypes

import numpy as np
import pytest

from helpers import REL_TOL, oracle_out, oracle_route, rel_l2
from workloads import configs, gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pw():
    import any_precision_bitplane_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.lib()
    return m


@pytest.mark.parametrize("spec", [("hb_dec", 256, 128, 8, 2, 12, 1), ("hb_pre", 256, 128, 4, 2, 600, 2)],
                         ids=["decode", "prefill"])
def test_host_buffers_match_device_buffers(pw, spec):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    name, H, I, E, k, T, path = spec
    layer = gen.make_layer(configs.custom(name, H, I, E, k, T), seed=81)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, k)
        h_hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16).copy()).pin_memory()
        h_ids = torch.from_numpy(ids).pin_memory()
        h_w = torch.from_numpy(w).pin_memory()
        h_out = torch.full((T, H), float("nan"), dtype=torch.float32).pin_memory()
        shape = pw.MoeShape(T, H, I, E, k)
        nbytes = pw.workspace_bytes(T, H, I, E, k)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        stream = torch.cuda.current_stream()
        rc = pw.lib().pw_moe_forward_path(
            ctypes.byref(shape), ctypes.c_void_p(h_hidden.data_ptr()),
            ctypes.c_void_p(h_ids.data_ptr()), ctypes.c_void_p(h_w.data_ptr()), dl.table.handle,
            ctypes.c_void_p(h_out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
            ctypes.c_size_t(nbytes), path, ctypes.c_void_p(stream.cuda_stream))
        assert rc == pw.PW_OK, pw.last_error()
        torch.cuda.synchronize()
        dev = pw.moe_forward(h_hidden.cuda(), h_ids.cuda(), h_w.cuda(), dl.table, dl.I, dl.E,
                             path=path).cpu()
        assert dl.table.status() == pw.PW_OK
        assert torch.equal(h_out, dev)
        assert rel_l2(h_out.numpy(), oracle_out(layer, tok.hidden_bf16, ids, w)) <= REL_TOL
    finally:
        dl.close()
