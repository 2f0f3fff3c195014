"""Routing statistics accumulated by forward calls (per-expert pair counts and
routing mass) against the oracle: counts bit-exact, mass to float tolerance
(the device sums with atomics in any order)."""
import numpy as np
import pytest

from helpers import oracle_route
from oracle import moe
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


CASES = [
    # name, H, I, E, k, T, path: decode, decode with GEMM-path experts, prefill
    ("dec", 256, 128, 12, 2, 9, 1, "normal"),
    ("hyb", 256, 128, 8, 2, 48, 1, "zipf"),
    ("pre", 256, 128, 4, 2, 600, 2, "normal"),
]


@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_stats_accumulate_over_calls(pw, spec):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    name, H, I, E, k, T, path, logits = spec
    layer = gen.make_layer(configs.custom(name, H, I, E, k, T, logit_mode=logits), seed=51)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, k)
        ids[1, 0] = E + 2          # an invalid id: left out of the statistics
        hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
        d_ids, d_w = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
        counts = torch.zeros(E, dtype=torch.int32, device="cuda")
        mass = torch.zeros(E, dtype=torch.float32, device="cuda")
        dl.table.set_routing_stats(counts, mass)
        for _ in range(2):
            pw.moe_forward(hidden, d_ids, d_w, dl.table, dl.I, dl.E, path=path)
        dl.table.set_routing_stats(None, None)
        pw.moe_forward(hidden, d_ids, d_w, dl.table, dl.I, dl.E, path=path)   # not counted
        torch.cuda.synchronize()
        assert dl.table.status() == pw.PW_ERR_BAD_EXPERT_ID
        c_ref, m_ref = moe.routing_stats(ids, w, E)
        np.testing.assert_array_equal(counts.cpu().numpy(), 2 * c_ref)
        np.testing.assert_allclose(mass.cpu().numpy(), 2 * m_ref, rtol=1e-5, atol=1e-6)
    finally:
        dl.close()


def test_stats_planner_recommit_end_to_end(pw):
    # routing statistics of one call feed the planner; its recommit list goes
    # through the page table, and the next call matches the oracle at the
    # planned bitwidths
    from any_precision_bitplane_gb300.layer import DeviceLayer
    from helpers import REL_TOL, oracle_out, rel_l2
    layer = gen.make_layer(configs.LayerConfig("plan", H=256, I=128, E=16, k=4, T=(32,),
                                               logit_mode="zipf"), 61)
    dl = DeviceLayer(layer)
    try:
        T, E = 32, 16
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, 4)
        args = (torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
                torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
        counts = torch.zeros(E, dtype=torch.int32, device="cuda")
        mass = torch.zeros(E, dtype=torch.float32, device="cuda")
        dl.table.set_routing_stats(counts, mass)
        pw.moe_forward(*args, dl.table, dl.I, dl.E)
        dl.table.set_routing_stats(None, None)
        mass_h = mass.cpu().numpy()
        q_now = dl.q.ravel().copy()
        bpb = np.array([2 * 128 * 256 // 8, 256 * 128 // 8] * E, dtype=np.int64)
        target = int(0.25 * (q_now * bpb).sum())
        sens = gen.make_sensitivity(layer)
        blocks, new_q, freed = pw.plan_recommit(q_now, sens, bpb, mass_h, 6, target)
        from oracle import planner
        assert (blocks, new_q, freed) == planner.plan_recommit(q_now.tolist(), sens, bpb.tolist(),
                                                               mass_h, 6, target)
        assert freed >= target and blocks
        dl.commit(blocks, new_q)
        got = pw.moe_forward(*args, dl.table, dl.I, dl.E).cpu().numpy()
        assert dl.table.status() == pw.PW_OK
        assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w, q=dl.q)) <= REL_TOL
        total = sum(float(m) for m in mass_h)
        hot = [float(m) * E > total for m in mass_h]
        assert all(q >= 6 for b, q in zip(blocks, new_q) if hot[b // 2])
    finally:
        dl.close()
