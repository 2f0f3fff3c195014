"""Decode calls where some experts hold many pairs: those experts run through
the tensor-core GEMM kernels (8 or more pairs, in calls of 16 or more tokens),
the rest through the decode kernels, and the two halves meet in the combine.

Checked against the oracle (2e-3 relative L2) and against the same call
through pw_moe_forward_noalloc, which keeps every expert on the decode
kernels: the two agree to tolerance but not bit for bit, which shows that the
GEMM kernels really took part."""
import ctypes

import numpy as np
import pytest

from helpers import REL_TOL, oracle_out, oracle_route, rel_l2
from workloads import configs, gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

HEAVY = 8    # pairs from which an expert goes to the GEMM kernels (calls of >= 16 tokens)


@pytest.fixture(scope="module")
def pw():
    import any_precision_bitplane_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.lib()
    return m


def _inputs(tok, ids, w):
    return (torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
            torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())


def _noalloc(pw, dl, k, hidden, ids, w):
    T = hidden.shape[0]
    out = torch.full((T, dl.H), float("nan"), dtype=torch.float32, device="cuda")
    shape = pw.MoeShape(T, dl.H, dl.I, dl.E, k)
    rc = pw.lib().pw_moe_forward_noalloc(
        ctypes.byref(shape), ctypes.c_void_p(hidden.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
        ctypes.c_void_p(w.data_ptr()), dl.table.handle, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pw.PW_OK, pw.last_error()
    return out.cpu().numpy()


SHAPES = [
    # name, H, I, E, k, T, logits: Zipf routing puts 8+ pairs on the first
    # experts (one of them exactly 8) and a few on the rest
    ("zipf_mix", 256, 128, 8, 2, 48, "zipf"),
    ("wide_tail", 128, 192, 16, 4, 40, "zipf"),
]


@pytest.mark.parametrize("spec", SHAPES, ids=[s[0] for s in SHAPES])
def test_heavy_and_light_experts(pw, spec):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    name, H, I, E, k, T, logit_mode = spec
    layer = gen.make_layer(configs.custom(name, H, I, E, k, T, logit_mode=logit_mode), seed=41)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, k)
        counts = np.bincount(ids.ravel(), minlength=E)
        assert counts.max() >= HEAVY and (counts[(counts > 0)] < HEAVY).any()
        args = _inputs(tok, ids, w)
        got = pw.moe_forward(*args, dl.table, dl.I, dl.E, path=pw.PATH_DECODE).cpu().numpy()
        assert dl.table.status() == pw.PW_OK
        ref = oracle_out(layer, tok.hidden_bf16, ids, w)
        assert rel_l2(got, ref) <= REL_TOL
        dec = _noalloc(pw, dl, k, *args)
        assert rel_l2(dec, ref) <= REL_TOL
        assert not np.array_equal(got, dec)
    finally:
        dl.close()


def test_every_expert_heavy(pw):
    # no expert is left to the decode kernels: the down launch only combines
    from any_precision_bitplane_gb300.layer import DeviceLayer
    T, k = 40, 1
    layer = gen.make_layer(configs.custom("all_heavy", 128, 64, 2, k, T), seed=42)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids = (np.arange(T, dtype=np.int32) % 2).reshape(T, k)
        w = np.ones((T, k), dtype=np.float32)
        got = pw.moe_forward(*_inputs(tok, ids, w), dl.table, dl.I, dl.E).cpu().numpy()
        assert dl.table.status() == pw.PW_OK
        assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w)) <= REL_TOL
    finally:
        dl.close()


def test_heavy_expert_not_resident_and_bad_id(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    name, H, I, E, k, T = "hv_err", 256, 128, 8, 2, 48
    layer = gen.make_layer(configs.custom(name, H, I, E, k, T, logit_mode="zipf"), seed=43)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, k)
        counts = np.bincount(ids.ravel(), minlength=E)
        heavy = int(np.argmax(counts))
        assert counts[heavy] >= HEAVY
        dl.table.set_pages([2 * heavy + 1], [dl.planes_ptr(2 * heavy + 1)], [pw.PW_PAGE_CPU])
        got = pw.moe_forward(*_inputs(tok, ids, w), dl.table, dl.I, dl.E).cpu().numpy()
        assert dl.table.status() == pw.PW_ERR_PAGE_NOT_RESIDENT
        ref = oracle_out(layer, tok.hidden_bf16, ids, w, drop_experts=[heavy])
        assert rel_l2(got, ref) <= REL_TOL
        dl.table.set_pages([2 * heavy + 1], [dl.planes_ptr(2 * heavy + 1)], [pw.PW_PAGE_GPU])
        bad = ids.copy()
        bad[0, 1] = E + 3
        w0 = w.copy()
        w0[0, 1] = 0.0
        got = pw.moe_forward(*_inputs(tok, bad, w), dl.table, dl.I, dl.E).cpu().numpy()
        assert dl.table.status() == pw.PW_ERR_BAD_EXPERT_ID
        assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w0)) <= REL_TOL
    finally:
        dl.close()
