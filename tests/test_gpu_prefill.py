"""The prefill path (dequantise into shared memory -> tcgen05 MMA) against the oracle.

Operands are fp16 (exact LUT weights, hidden states converted from bf16), h is
fp16, accumulation fp32: the output is held to the same 2e-3 relative L2 as
the decode path."""
import dataclasses

import numpy as np
import pytest

from helpers import REL_TOL, host_layer, oracle_out, oracle_out_pool, oracle_route, rel_l2
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


def _run(pw, dl, tok, ids, w, path):
    hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
    out = pw.moe_forward(hidden, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                         dl.table, dl.I, dl.E, path=path)
    return out.cpu().numpy(), dl.table.status()


SHAPES = [
    # name, H, I, E, k, T: token tiles of 256 with ragged tails, several row tiles
    ("p_small", 256, 128, 4, 2, 300),
    ("p_two_tiles", 128, 192, 2, 1, 700),
    ("p_many_experts", 256, 64, 16, 4, 257),
    ("p_single", 128, 64, 1, 1, 5),
]


@pytest.mark.parametrize("spec", SHAPES, ids=[s[0] for s in SHAPES])
def test_prefill_small_shapes(pw, spec):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    name, H, I, E, k, T = spec
    layer = gen.make_layer(configs.custom(name, H, I, E, k, T), seed=31)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, k)
        got, status = _run(pw, dl, tok, ids, w, pw.PATH_PREFILL)
        assert status == pw.PW_OK
        ref = oracle_out(layer, tok.hidden_bf16, ids, w)
        assert rel_l2(got, ref) <= REL_TOL
    finally:
        dl.close()


@pytest.mark.parametrize("q", [3, 4, 5, 6, 8])
def test_prefill_each_bitwidth(pw, q):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = gen.make_layer(configs.custom("pq", 256, 128, 3, 2, 200), seed=32)
    layer = dataclasses.replace(layer, q=np.full_like(layer.q, q))
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, 200)
        ids, w = oracle_route(tok, 2)
        got, status = _run(pw, dl, tok, ids, w, pw.PATH_PREFILL)
        assert status == pw.PW_OK
        assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w)) <= REL_TOL
    finally:
        dl.close()


def test_prefill_and_decode_agree(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = gen.make_layer(configs.custom("pd", 256, 256, 8, 2, 600), seed=33)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, 600)
        ids, w = oracle_route(tok, 2)
        pre, s1 = _run(pw, dl, tok, ids, w, pw.PATH_PREFILL)
        dec, s2 = _run(pw, dl, tok, ids, w, pw.PATH_DECODE)
        assert s1 == pw.PW_OK and s2 == pw.PW_OK
        assert rel_l2(pre, dec) <= REL_TOL
        # automatic path choice takes prefill here
        assert 600 * 2 >= pw.prefill_min_pairs(600, 256, 256, 8, 2)
    finally:
        dl.close()


def test_prefill_skips_non_resident_and_bad_ids(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = gen.make_layer(configs.custom("pf", 256, 128, 4, 2, 300), seed=34)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, 300)
        ids, w = oracle_route(tok, 2)
        e = int(ids[0, 0])
        dl.table.set_pages([2 * e], [dl.planes_ptr(2 * e)], [pw.PW_PAGE_IN_TRANSFER])
        got, status = _run(pw, dl, tok, ids, w, pw.PATH_PREFILL)
        assert status == pw.PW_ERR_PAGE_NOT_RESIDENT
        ref = oracle_out(layer, tok.hidden_bf16, ids, w, drop_experts=[e])
        assert rel_l2(got, ref) <= REL_TOL
        dl.table.set_pages([2 * e], [dl.planes_ptr(2 * e)], [pw.PW_PAGE_GPU])
        bad = ids.copy()
        bad[5, 1] = 99
        w0 = w.copy()
        w0[5, 1] = 0.0
        got, status = _run(pw, dl, tok, bad, w, pw.PATH_PREFILL)
        assert status == pw.PW_ERR_BAD_EXPERT_ID
        assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w0)) <= REL_TOL
    finally:
        dl.close()


def test_prefill_rejects_unsupported_shape(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = gen.make_layer(configs.custom("pbad", 96, 64, 2, 1, 8), seed=35)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, 8)
        ids, w = oracle_route(tok, 1)
        with pytest.raises(pw.PWError) as ei:
            _run(pw, dl, tok, ids, w, pw.PATH_PREFILL)
        assert ei.value.code == pw.PW_ERR_SHAPE
        # the automatic choice never picks prefill for it
        assert pw.prefill_min_pairs(8, 96, 64, 2, 1) > 2**30
    finally:
        dl.close()


def test_mixtral_prefill_full_output(pw):
    # full-size Mixtral-shaped prefill (4096 tokens, 8 experts, top-2) through
    # the automatic path, checked on every token: the oracle computes all
    # 4096 outputs (8 experts' blocks dequantised in fp64, a spawn pool), and
    # the error is held per token, so that no token tile of any expert can
    # hide inside a pooled norm
    from any_precision_bitplane_gb300.layer import DeviceLayer
    name = "mixtral_prefill"
    layer = host_layer(name)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, 4096)
        ids, w = oracle_route(tok, 2)
        got, status = _run(pw, dl, tok, ids, w, pw.PATH_AUTO)
        assert status == pw.PW_OK
        assert np.isfinite(got).all()
    finally:
        dl.close()
    ref = oracle_out_pool(name, tok.hidden_bf16, ids, w, layer.q, workers=8)
    assert rel_l2(got, ref) <= REL_TOL
    per_token = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert per_token.max() <= REL_TOL, (int(per_token.argmax()), float(per_token.max()))
