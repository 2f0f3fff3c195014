"""Router and token-to-expert permutation on the GPU against the oracle.

Ids and the permutation are integer results: bit-exact.  Router weights are
fp32 softmax values over the kept logits: relative error <= 1e-6."""
import numpy as np
import pytest

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


def _logits(cfg_name, T):
    cfg = configs.config_by_name(cfg_name)
    # the router sees only logits: draw them with the layer's recipe on a tiny layer
    small = configs.LayerConfig(cfg.name, H=32, I=32, E=cfg.E, k=cfg.k, T=(T,),
                                q_mode=cfg.q_mode, logit_mode=cfg.logit_mode, hot=cfg.hot)
    return gen.make_tokens(gen.make_layer(small, 0), T).logits, cfg


@pytest.mark.parametrize("name,T", [("tiny", 16), ("qwen15_decode", 8), ("mixtral_decode", 4),
                                    ("qwen3_decode", 64), ("mixtral_prefill", 4096)])
def test_route_topk_matches_oracle(pw, name, T):
    logits, cfg = _logits(name, T)
    ids, w = pw.route_topk(torch.from_numpy(logits).cuda(), cfg.k)
    ref_ids, ref_w = moe.route_topk(logits, cfg.k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=1e-6, atol=1e-7)


def test_route_ties_and_extremes(pw):
    logits = np.array([[1.0, 3.0, 3.0, 3.0, 0.0, -np.inf],
                       [-np.inf, -np.inf, -np.inf, -np.inf, 5.0, -np.inf],
                       [0.0, 0.0, 0.0, 0.0, 0.0, 0.0]], np.float32)
    ids, w = pw.route_topk(torch.from_numpy(logits).cuda(), 2)
    ref_ids, ref_w = moe.route_topk(logits, 2)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("E,T,k", [(8, 16, 2), (60, 8, 4), (128, 64, 8), (8, 4096, 2),
                                   (1024, 300, 5), (3, 1, 1), (1, 7, 1)])
def test_permute_bit_exact(pw, E, T, k):
    rng = np.random.default_rng(E * 7 + T)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    off, perm, inv = pw.permute(torch.from_numpy(ids).cuda(), E)
    r_off, r_perm, r_inv = moe.permute(ids, E)
    np.testing.assert_array_equal(off.cpu().numpy(), r_off)
    np.testing.assert_array_equal(perm.cpu().numpy(), r_perm)
    np.testing.assert_array_equal(inv.cpu().numpy(), r_inv)


def test_permute_skewed_routing(pw):
    # Zipf-like skew: most pairs to expert 0, with repeated ids inside a token
    rng = np.random.default_rng(5)
    ids = np.where(rng.random((500, 4)) < 0.7, 0, rng.integers(0, 16, (500, 4))).astype(np.int32)
    off, perm, inv = pw.permute(torch.from_numpy(ids).cuda(), 16)
    r_off, r_perm, r_inv = moe.permute(ids, 16)
    np.testing.assert_array_equal(off.cpu().numpy(), r_off)
    np.testing.assert_array_equal(perm.cpu().numpy(), r_perm)


def test_permute_long_runs_per_warp(pw):
    # 40000 pairs: every warp of the permute CTA walks ~40 steps of 32 pairs,
    # so each expert's running start carries across many steps; heavy skew
    # puts up to 32 lanes of one step on the same expert
    rng = np.random.default_rng(11)
    ids = np.where(rng.random((20000, 2)) < 0.5, rng.integers(0, 3, (20000, 2)),
                   rng.integers(0, 64, (20000, 2))).astype(np.int32)
    off, perm, inv = pw.permute(torch.from_numpy(ids).cuda(), 64)
    r_off, r_perm, r_inv = moe.permute(ids, 64)
    np.testing.assert_array_equal(off.cpu().numpy(), r_off)
    np.testing.assert_array_equal(perm.cpu().numpy(), r_perm)
    np.testing.assert_array_equal(inv.cpu().numpy(), r_inv)


def test_permute_empty(pw):
    ids = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    off, perm, inv = pw.permute(ids, 5)
    assert off.cpu().tolist() == [0] * 6 and perm.numel() == 0


def test_permute_bad_ids_latch_status_and_drop(pw):
    ids = np.array([[0, 9], [2, -1], [2, 1]], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    off, perm, inv = pw.permute(torch.from_numpy(ids).cuda(), 4, status=status)
    assert status.item() == pw.PW_ERR_BAD_EXPERT_ID
    assert off.cpu().tolist() == [0, 1, 2, 4, 4]
    assert perm.cpu().numpy()[:4].tolist() == [0, 5, 2, 4]
    inv = inv.cpu().numpy()
    assert inv[1] == -1 and inv[3] == -1 and inv[0] == 0 and inv[5] == 1
