"""pw_moe_forward_logits: the router fused into the launch that groups the
pairs (PagedWeight, "Core components" 3: one fused operation; "Core
components" 2: the routing weights are the mass the planner tracks).

On every workload the fused call must route exactly as the oracle's router
(ids bit for bit, weights to 1e-6), and its output must be bit-identical to
the separate router launch followed by pw_moe_forward (both are
deterministic); on the smaller workloads it is also held to the oracle's
layer output."""
import numpy as np
import pytest

from helpers import REL_TOL, host_layer, oracle_out, oracle_route, rel_l2
from oracle import moe
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


CASES = [("tiny", 16, True), ("qwen15_decode", 1, True), ("qwen15_decode", 4, True),
         ("qwen15_decode", 8, True), ("qwen3_decode", 64, True), ("mixtral_decode", 4, False),
         ("mixtral_prefill", 4096, False)]


@pytest.mark.parametrize("name,T,with_oracle", CASES, ids=["%s-T%d" % (c[0], c[1]) for c in CASES])
def test_fused_router_forward(pw, name, T, with_oracle):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = host_layer(name)
    cfg = layer.cfg
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
        logits = torch.from_numpy(tok.logits).cuda()
        out, ids, wts = pw.moe_forward_logits(hidden, logits, dl.table, cfg.I, cfg.E, cfg.k)
        torch.cuda.synchronize()
        assert dl.table.status() == pw.PW_OK
        # the separate router and the plain entry point, for bit identity
        ids2, wts2 = pw.route_topk(logits, cfg.k)
        out2 = pw.moe_forward(hidden, ids2, wts2, dl.table, cfg.I, cfg.E)
        got, got_ids, got_w = out.cpu().numpy(), ids.cpu().numpy(), wts.cpu().numpy()
        assert np.array_equal(got_ids, ids2.cpu().numpy())
        assert np.array_equal(got_w, wts2.cpu().numpy())
        assert np.array_equal(got, out2.cpu().numpy())
    finally:
        dl.close()
    ref_ids, ref_w = moe.route_topk(tok.logits, cfg.k)
    assert np.array_equal(got_ids, ref_ids)
    assert np.max(np.abs(got_w - ref_w) / ref_w) <= 1e-6
    if with_oracle:
        ids_o, w_o = oracle_route(tok, cfg.k)
        ref = oracle_out(layer, tok.hidden_bf16, ids_o, w_o)
        assert rel_l2(got, ref) <= REL_TOL


def test_fused_router_routing_statistics(pw):
    # the routing statistics by-product sees the fused router's output
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = host_layer("qwen3_decode")
    cfg = layer.cfg
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, 64)
        counts = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
        mass = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
        dl.table.set_routing_stats(counts, mass)
        _, ids, wts = pw.moe_forward_logits(torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
                                            torch.from_numpy(tok.logits).cuda(), dl.table, cfg.I,
                                            cfg.E, cfg.k)
        torch.cuda.synchronize()
        dl.table.set_routing_stats(None, None)
        want_c, want_m = moe.routing_stats(ids.cpu().numpy(), wts.cpu().numpy(), cfg.E)
        assert np.array_equal(counts.cpu().numpy(), want_c)
        np.testing.assert_allclose(mass.cpu().numpy(), want_m, rtol=1e-5, atol=1e-6)
    finally:
        dl.close()


def test_fused_router_rejects_null_logits(pw):
    layer = host_layer("tiny")
    from any_precision_bitplane_gb300.layer import DeviceLayer
    dl = DeviceLayer(layer)
    try:
        import ctypes
        s = pw.MoeShape(4, layer.cfg.H, layer.cfg.I, layer.cfg.E, layer.cfg.k)
        rc = pw.lib().pw_moe_forward_logits(ctypes.byref(s), None, None, None, None, dl.table.handle,
                                            None, None, 0, 0, None)
        assert rc == pw.PW_ERR_INVALID_ARG
    finally:
        dl.close()
