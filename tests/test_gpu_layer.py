"""The fused layer (pw_moe_forward) on the GPU against the CPU oracle.

Tolerance: relative L2 error of the fp32 output <= 2e-3 (REL_TOL).  Inputs:
the seeded workloads; routing from the oracle's router so that both sides see
identical topk ids and weights."""
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


_DEV = {}


def device_layer(layer, key):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    if key not in _DEV:
        if len(_DEV) >= 2:
            for v in _DEV.values():
                v.close()
            _DEV.clear()
            torch.cuda.empty_cache()
        _DEV[key] = DeviceLayer(layer)
    return _DEV[key]


def run(pw, dl, hidden_bits, ids, w, path=0):
    hidden = torch.from_numpy(hidden_bits.view(np.int16)).cuda()
    out = pw.moe_forward(hidden, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                         dl.table, dl.I, dl.E, path=path)
    got = out.cpu().numpy()
    return got, dl.table.status()


def check(pw, layer, key, T, path=0, q=None):
    dl = device_layer(layer, key)
    tok = gen.make_tokens(layer, T)
    ids, w = oracle_route(tok, layer.cfg.k)
    got, status = run(pw, dl, tok.hidden_bf16, ids, w, path)
    assert status == pw.PW_OK
    ref = oracle_out(layer, tok.hidden_bf16, ids, w, q=q)
    err = rel_l2(got, ref)
    assert err <= REL_TOL, err
    return err


def test_tiny_config(pw):
    layer = host_layer("tiny")
    check(pw, layer, "tiny", 16)


CUSTOM = [
    # name, H, I, E, k, T -- ragged splits of K over the 8 warps, empty warps,
    # k = E, token groups beyond 8, single token / single expert
    ("one", 32, 32, 1, 1, 1),
    ("ragged", 64, 96, 3, 2, 5),
    ("wideH", 160, 64, 4, 2, 9),
    ("allexp", 256, 512, 8, 8, 3),
    ("manytok", 96, 160, 2, 1, 37),
    # long down blocks (I >= 8192): the down tiles split K in two parts; 257
    # words split 128/129 and raggedly over the warps, H = 96 leaves a
    # 32-row last range
    ("ksplit", 96, 8224, 3, 2, 3),
]


@pytest.mark.parametrize("spec", CUSTOM, ids=[c[0] for c in CUSTOM])
def test_custom_shapes(pw, spec):
    name, H, I, E, k, T = spec
    layer = gen.make_layer(configs.custom(name, H, I, E, k, T), seed=21)
    check(pw, layer, name, T)


@pytest.mark.parametrize("q", [3, 4, 5, 6, 8])
def test_uniform_bitwidth(pw, q):
    layer = gen.make_layer(configs.custom("uq", 256, 192, 6, 2, 12), seed=22)
    layer = dataclasses.replace(layer, q=np.full_like(layer.q, q))
    check(pw, layer, "uq%d" % q, 12)


@pytest.mark.parametrize("q", [3, 4, 5, 6, 8])
def test_ksplit_uniform_bitwidth(pw, q):
    # every table form of the down tiles with K split in two parts
    layer = gen.make_layer(configs.custom("ksq", 96, 8224, 3, 2, 3), seed=24)
    layer = dataclasses.replace(layer, q=np.full_like(layer.q, q))
    check(pw, layer, "ksq%d" % q, 3)


@pytest.mark.parametrize("q", [3, 4, 5, 6, 8])
def test_long_gateup_k_uniform_bitwidth(pw, q):
    # H = 4096: 16 word columns per warp in every gate_up pass, I = 96 a
    # ragged last tile
    layer = gen.make_layer(configs.custom("lk", 4096, 96, 4, 2, 5), seed=25)
    layer = dataclasses.replace(layer, q=np.full_like(layer.q, q))
    check(pw, layer, "lk%d" % q, 5)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_qwen15_decode(pw, T):
    check(pw, host_layer("qwen15_decode"), "qwen15_decode", T)


def test_qwen3_decode(pw):
    check(pw, host_layer("qwen3_decode"), "qwen3_decode", 64)


def test_mixtral_decode(pw):
    name = "mixtral_decode"
    layer = host_layer(name)
    dl = device_layer(layer, name)
    tok = gen.make_tokens(layer, 4)
    ids, w = oracle_route(tok, layer.cfg.k)
    got, status = run(pw, dl, tok.hidden_bf16, ids, w)
    assert status == pw.PW_OK
    ref = oracle_out_pool(name, tok.hidden_bf16, ids, w, layer.q)
    assert rel_l2(got, ref) <= REL_TOL


def test_fused_mixed_launch_equals_sum_of_single_expert_calls(pw):
    # One launch over blocks of different bitwidths equals the sum of launches
    # that each see one expert (its other top-k weights set to zero).
    layer = host_layer("tiny")
    dl = device_layer(layer, "tiny")
    tok = gen.make_tokens(layer, 16)
    ids, w = oracle_route(tok, layer.cfg.k)
    fused, _ = run(pw, dl, tok.hidden_bf16, ids, w)
    total = np.zeros_like(fused, dtype=np.float64)
    for e in np.unique(ids):
        w_e = np.where(ids == e, w, 0).astype(np.float32)
        part, _ = run(pw, dl, tok.hidden_bf16, ids, w_e)
        total += part
    assert rel_l2(fused, total) <= 1e-5
    assert len(set(int(v) for v in layer.q.ravel())) > 1   # the launch really mixed bitwidths


def test_ksplit_forward_is_repeatable(pw):
    # the two K parts' partial sums are added in a fixed order by the combine
    layer = gen.make_layer(configs.custom("ksplit_rep", 96, 8224, 3, 2, 3), seed=23)
    dl = device_layer(layer, "ksplit_rep")
    tok = gen.make_tokens(layer, 3)
    ids, w = oracle_route(tok, layer.cfg.k)
    a, sa = run(pw, dl, tok.hidden_bf16, ids, w)
    b, sb = run(pw, dl, tok.hidden_bf16, ids, w)
    assert sa == sb == pw.PW_OK
    np.testing.assert_array_equal(a, b)


def test_forward_is_repeatable(pw):
    layer = host_layer("tiny")
    dl = device_layer(layer, "tiny")
    tok = gen.make_tokens(layer, 16)
    ids, w = oracle_route(tok, layer.cfg.k)
    a, _ = run(pw, dl, tok.hidden_bf16, ids, w)
    b, _ = run(pw, dl, tok.hidden_bf16, ids, w)
    np.testing.assert_array_equal(a, b)   # no atomics on the output: deterministic


def test_zero_tokens(pw):
    layer = host_layer("tiny")
    dl = device_layer(layer, "tiny")
    hidden = torch.zeros((0, layer.cfg.H), dtype=torch.int16, device="cuda")
    ids = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    w = torch.zeros((0, 2), dtype=torch.float32, device="cuda")
    out = pw.moe_forward(hidden, ids, w, dl.table, dl.I, dl.E)
    assert out.shape == (0, layer.cfg.H)


def test_workspace_too_small_is_rejected(pw):
    layer = host_layer("tiny")
    dl = device_layer(layer, "tiny")
    tok = gen.make_tokens(layer, 16)
    ids, w = oracle_route(tok, layer.cfg.k)
    hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pw.PWError) as ei:
        pw.moe_forward(hidden, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                       dl.table, dl.I, dl.E, workspace=ws)
    assert ei.value.code == pw.PW_ERR_WORKSPACE


def test_back_to_back_calls_of_mixed_sizes_share_one_workspace(pw):
    # Calls of different sizes queued on one stream with no host sync between
    # them, all on one workspace: small calls (whose down grid leaves SM slots
    # free) launch their grouping kernel early, behind the previous call's
    # down kernel; large calls launch it plainly.  Every transition must leave
    # each call's result equal to the oracle's.
    layer = gen.make_layer(configs.custom("mixed_sizes", 1024, 256, 32, 4, 64), seed=31)
    dl = device_layer(layer, "mixed_sizes")
    sizes = [1, 64, 1, 2, 64, 1, 3]
    ws = torch.empty(max(pw.workspace_bytes(T, dl.H, dl.I, dl.E, 4) for T in sizes),
                     dtype=torch.uint8, device="cuda")
    # each call takes its own slice of one token stream, so inputs differ
    pool = gen.make_tokens(layer, sum(sizes))
    calls, t0 = [], 0
    for T in sizes:
        tok = gen.Tokens(pool.hidden_bf16[t0:t0 + T].copy(), pool.logits[t0:t0 + T].copy())
        t0 += T
        ids, w = oracle_route(tok, 4)
        args = (torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
                torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
        calls.append((tok, ids, w, args))
    torch.cuda.synchronize()
    outs = [pw.moe_forward(*args, dl.table, dl.I, dl.E, workspace=ws) for _, _, _, args in calls]
    torch.cuda.synchronize()
    assert dl.table.status() == pw.PW_OK
    for (tok, ids, w, _), out in zip(calls, outs):
        ref = oracle_out(layer, tok.hidden_bf16, ids, w)
        assert rel_l2(out.cpu().numpy(), ref) <= REL_TOL
