"""Pins for the CPU oracle, checked against things other than the oracle itself.

Each test names what fixes the expected value: a worked example under
tests/golden/, a closed form, an identity the format guarantees, a library
routine, or an independent brute force.
"""
import math
import os

import numpy as np
import pytest

from oracle import apl, moe, planner
from workloads import configs, gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- bitplanes

def test_pack_worked_example():
    rows = _read_golden("bitplane_worked_example.txt")
    codes = np.zeros((2, 64), np.uint8)
    want = np.zeros((8, 2, 2), np.uint32)            # [plane][word][row]
    for r in rows:
        if r[0] == "code":
            codes[int(r[1]), int(r[2])] = int(r[3])
        elif r[0] == "plane":
            want[int(r[1]), int(r[3]), int(r[2])] = int(r[4], 16)
    got = apl.pack_bitplanes(codes)
    np.testing.assert_array_equal(got, want)
    for r in rows:
        if r[0] == "idx":
            b, n, k, v = map(int, r[1:])
            assert int(apl.unpack_top(got, b)[n, k]) == v, r


@pytest.mark.parametrize("shape", [(1, 32), (3, 96), (17, 64), (64, 256)])
def test_unpack_top_equals_code_shift(shape):
    # identity fixed by the format: the top-b planes give code >> (8-b), all b
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=shape, dtype=np.uint8)
    planes = apl.pack_bitplanes(codes)
    for b in range(1, 9):
        np.testing.assert_array_equal(apl.unpack_top(planes, b), codes >> (8 - b))


def test_planes_are_a_prefix():
    # the b-bit view must not depend on planes b..7 (they can be freed)
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, size=(8, 64), dtype=np.uint8)
    planes = apl.pack_bitplanes(codes)
    for b in (3, 4, 5, 6):
        trunc = planes.copy()
        trunc[b:] = rng.integers(0, 2**32, size=trunc[b:].shape, dtype=np.uint64).astype(np.uint32)
        np.testing.assert_array_equal(apl.unpack_top(trunc, b), codes >> (8 - b))


def test_pack_bit_population():
    # each plane carries exactly the population of its code bit
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, size=(5, 128), dtype=np.uint8)
    planes = apl.pack_bitplanes(codes)
    for p in range(8):
        pop = sum(bin(int(w)).count("1") for w in planes[p].ravel())
        assert pop == int(((codes >> (7 - p)) & 1).sum())


def test_pack_rejects_ragged_k():
    with pytest.raises(ValueError):
        apl.pack_bitplanes(np.zeros((2, 48), np.uint8))


# ---------------------------------------------------------------- dequant

def test_dequant_worked_example():
    rows = _read_golden("lut_worked_example.txt")
    lut = None
    for r in rows:
        if r[0] == "lut":
            lut = np.array([float(v) for v in r[2:]], np.float16)[None, :]
    assert lut is not None
    for r in rows:
        if r[0] == "weight":
            q, code, w = int(r[1]), int(r[2]), float(r[3])
            codes = np.full((1, 32), code, np.uint8)
            got = apl.dequant(apl.pack_bitplanes(codes), lut, q)
            assert np.all(got == w), r


def test_dequant_b8_reproduces_lut_weights():
    # spec invariant: q = 8 gives the full-precision LUT weights
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 256, size=(12, 64), dtype=np.uint8)
    lut8 = np.sort(rng.normal(0, 0.02, (12, 256)).astype(np.float16), axis=1)
    got = apl.dequant(apl.pack_bitplanes(codes), lut8, 8)
    want = np.array([[float(lut8[n, codes[n, k]]) for k in range(64)] for n in range(12)])
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("q", [3, 4, 5, 6, 8])
def test_dequant_integer_and_row_tagged_luts(q):
    # closed form: LUT_q[n][v] = 1000 n + v gives 1000 n + (code >> (8-q))
    rng = np.random.default_rng(7 + q)
    N, K = 6, 96
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    lut = (1000.0 * np.arange(N)[:, None] + np.arange(1 << q)[None, :])
    got = apl.dequant(apl.pack_bitplanes(codes), lut, q)
    want = 1000.0 * np.arange(N)[:, None] + (codes >> (8 - q))
    np.testing.assert_array_equal(got, want)


def test_dequant_rejects_wrong_lut_width():
    with pytest.raises(ValueError):
        apl.dequant(apl.pack_bitplanes(np.zeros((1, 32), np.uint8)), np.zeros((1, 16)), 3)


# ---------------------------------------------------------------- routing

def _brute_topk(row, k):
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(row):
            if e in chosen:
                continue
            if best is None or v > row[best]:      # strict: lower id wins ties
                best = e
        chosen.append(best)
    return chosen


def test_route_topk_selection_and_renormalisation():
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((40, 16)).astype(np.float32)
    ids, w = moe.route_topk(logits, 4)
    for t in range(40):
        assert list(ids[t]) == _brute_topk([float(v) for v in logits[t]], 4)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_route_topk_closed_forms():
    logits = np.array([[0.5, 2.0, -1.0, 1.0]], np.float32)
    ids, w = moe.route_topk(logits, 1)
    assert ids.tolist() == [[1]] and w.tolist() == [[1.0]]
    ids, w = moe.route_topk(logits, 2)
    assert ids.tolist() == [[1, 3]]
    # two kept experts: w0 / w1 = exp(l0 - l1)
    assert math.isclose(w[0, 0] / w[0, 1], math.exp(1.0), rel_tol=1e-13)
    assert math.isclose(w[0, 0], 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-13)


def test_route_topk_ties_go_to_lower_id():
    logits = np.array([[1.0, 3.0, 3.0, 3.0, 0.0]], np.float32)
    ids, w = moe.route_topk(logits, 2)
    assert ids.tolist() == [[1, 2]]
    np.testing.assert_allclose(w, [[0.5, 0.5]], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- permute

def test_permute_matches_bucket_loop():
    rng = np.random.default_rng(9)
    E, T, k = 7, 23, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    offsets, perm, inv = moe.permute(ids, E)
    buckets = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            buckets[int(ids[t, j])].append(t * k + j)
    flat = [p for b in buckets for p in b]
    assert perm.tolist() == flat
    start = 0
    for e in range(E):
        assert offsets[e] == start
        start += len(buckets[e])
    assert offsets[E] == T * k
    assert np.all(inv[perm] == np.arange(T * k))


def test_permute_empty_and_out_of_range():
    offsets, perm, inv = moe.permute(np.zeros((0, 2), np.int32), 4)
    assert offsets.tolist() == [0, 0, 0, 0, 0] and perm.size == 0 and inv.size == 0
    with pytest.raises(ValueError):
        moe.permute(np.array([[0, 4]], np.int32), 4)


def test_routing_stats_brute_force_and_invariants():
    # brute force: a plain loop over the pairs; invariants: every valid pair
    # counted once, and the renormalised router weights of a token sum to 1,
    # so the total routing mass equals the number of tokens
    rng = np.random.default_rng(7)
    T, E, k = 37, 9, 3
    ids, w = moe.route_topk(rng.standard_normal((T, E)), k)
    counts, mass = moe.routing_stats(ids, w, E)
    c_ref, m_ref = [0] * E, [0.0] * E
    for t in range(T):
        for j in range(k):
            c_ref[int(ids[t, j])] += 1
            m_ref[int(ids[t, j])] += float(w[t, j])
    assert counts.tolist() == c_ref
    np.testing.assert_allclose(mass, m_ref, rtol=1e-12)
    assert counts.sum() == T * k
    assert math.isclose(mass.sum(), T, rel_tol=1e-12)


def test_routing_stats_skips_out_of_range_ids():
    ids = np.array([[0, 5], [-1, 2]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    counts, mass = moe.routing_stats(ids, w, 4)
    assert counts.tolist() == [1, 0, 1, 0]
    assert mass.tolist() == [0.25, 0.0, 0.5, 0.0]


# ---------------------------------------------------------------- SiLU

def test_silu_textbook_values():
    for r in _read_golden("silu_values.txt"):
        g, v = float(r[1]), float(r[2])
        assert math.isclose(float(moe.silu(np.float64(g))), v, rel_tol=1e-15, abs_tol=1e-300)


# ---------------------------------------------------------------- parity metric

def test_rel_l2_closed_forms():
    # the metric every GPU parity test uses, pinned by values worked by hand
    # from its definition (tests/golden/rel_l2_closed_forms.txt)
    with open(os.path.join(GOLDEN, "rel_l2_closed_forms.txt")) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(lines) >= 8
    for ln in lines:
        got, ref, want = (part.split() for part in ln.split("|"))
        got = np.array([float(v) for v in got])
        ref = np.array([float(v) for v in ref])
        assert math.isclose(moe.rel_l2(got, ref), float(want[0]), rel_tol=1e-12, abs_tol=1e-15), ln


def test_rel_l2_scales_and_shapes():
    # scale invariance, 2-D tensors, and eps * ref giving exactly eps
    rng = np.random.default_rng(9)
    ref = rng.standard_normal((7, 5))
    for eps in (1e-6, 2e-3, 0.5):
        assert math.isclose(moe.rel_l2(ref * (1 + eps), ref), eps, rel_tol=1e-9)
        assert math.isclose(moe.rel_l2(1e8 * ref * (1 + eps), 1e8 * ref), eps, rel_tol=1e-9)
    # the error is pooled over the whole tensor, not averaged per row
    got = ref.copy()
    got[3] += 1.0
    want = math.sqrt(5.0) / math.sqrt(float((ref ** 2).sum()))
    assert math.isclose(moe.rel_l2(got, ref), want, rel_tol=1e-12)


# ---------------------------------------------------------------- full layer

def _layer_blocks(layer):
    cache = {}

    def block(e, m):
        if (e, m) not in cache:
            codes, luts, q = layer.block(e, m)
            cache[(e, m)] = (apl.pack_bitplanes(codes), luts[q], q)
        return cache[(e, m)]
    return block


def _brute_force_layer(layer, hidden_bits, ids, wts):
    """Explicit loops in Python floats, weights taken from the codes directly."""
    cfg = layer.cfg
    H, I = cfg.H, cfg.I
    T, k = ids.shape
    x = [[float(v) for v in row] for row in gen.bf16_bits_to_float32(hidden_bits)]

    def weight(e, m, n, kk):
        codes, luts, q = layer.block(e, m)
        return float(luts[q][n, int(codes[n, kk]) >> (8 - q)])

    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            h = []
            for i in range(I):
                g = sum(x[t][kk] * weight(e, 0, i, kk) for kk in range(H))
                u = sum(x[t][kk] * weight(e, 0, I + i, kk) for kk in range(H))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for n in range(H):
                y = sum(h[i] * weight(e, 1, n, i) for i in range(I))
                out[t][n] += float(wts[t, j]) * y
    return np.array(out)


def test_moe_forward_matches_brute_force():
    cfg = configs.custom("brute", H=64, I=32, E=4, k=2, T=3)
    layer = gen.make_layer(cfg, seed=11)
    tok = gen.make_tokens(layer, 3)
    ids, w = moe.route_topk(tok.logits, cfg.k)
    w32 = w.astype(np.float32)
    got = moe.moe_forward(tok.hidden_bf16, ids, w32, _layer_blocks(layer), cfg.E)
    want = _brute_force_layer(layer, tok.hidden_bf16, ids, w32)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-14)
    assert moe.rel_l2(got, want) < 1e-12


def test_moe_forward_token_subset_matches_full():
    cfg = configs.custom("subset", H=64, I=64, E=5, k=2, T=9)
    layer = gen.make_layer(cfg, seed=12)
    tok = gen.make_tokens(layer, 9)
    ids, w = moe.route_topk(tok.logits, cfg.k)
    blocks = _layer_blocks(layer)
    full = moe.moe_forward(tok.hidden_bf16, ids, w, blocks, cfg.E)
    part = moe.moe_forward(tok.hidden_bf16, ids, w, blocks, cfg.E, tokens=[2, 5, 8])
    np.testing.assert_allclose(part, full[[2, 5, 8]], rtol=1e-12, atol=1e-18)


def test_moe_forward_single_expert_weight_one_is_expert_output():
    # closed form: k = 1 and weight 1 give out = y_e exactly
    cfg = configs.custom("k1", H=32, I=32, E=3, k=1, T=2)
    layer = gen.make_layer(cfg, seed=13)
    tok = gen.make_tokens(layer, 2)
    ids = np.array([[2], [0]], np.int32)
    blocks = _layer_blocks(layer)
    out = moe.moe_forward(tok.hidden_bf16, ids, np.ones((2, 1), np.float32), blocks, cfg.E)
    x = moe.bf16_to_float64(tok.hidden_bf16)
    for t, e in ((0, 2), (1, 0)):
        w_gu = apl.dequant(*blocks(e, 0))
        w_dn = apl.dequant(*blocks(e, 1))
        np.testing.assert_array_equal(out[t], moe.expert_mlp(x[t:t + 1], w_gu, w_dn)[0])


def test_moe_forward_constant_luts_closed_form():
    # closed form: every gate/up weight c_g/c_u, every down weight c_d gives
    # out[t, n] = sum_j w_tj * I * SiLU(c_g S) * (c_u S) * c_d with S = sum_k x[t, k]
    cfg = configs.custom("const", H=64, I=32, E=2, k=2, T=2)
    layer = gen.make_layer(cfg, seed=14)
    tok = gen.make_tokens(layer, 2)
    c_g, c_u, c_d = 0.015625, -0.03125, 0.0078125

    def block(e, m):
        codes, _, q = layer.block(e, m)
        N = codes.shape[0]
        lut = np.full((N, 1 << q), c_d, np.float16)
        if m == 0:
            lut[:cfg.I] = c_g
            lut[cfg.I:] = c_u
        return apl.pack_bitplanes(codes), lut, q

    ids = np.array([[0, 1], [1, 0]], np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5]], np.float32)
    out = moe.moe_forward(tok.hidden_bf16, ids, w, block, cfg.E)
    S = moe.bf16_to_float64(tok.hidden_bf16).sum(axis=1)
    for t in range(2):
        g, u = c_g * S[t], c_u * S[t]
        val = cfg.I * (g / (1 + math.exp(-g))) * u * c_d
        np.testing.assert_allclose(out[t], val, rtol=1e-12)


def test_moe_forward_one_hot_hidden_picks_columns():
    # closed form: x = e_c gives g_i = W_gate[i, c], u_i = W_up[i, c]
    cfg = configs.custom("onehot", H=64, I=32, E=2, k=1, T=1)
    layer = gen.make_layer(cfg, seed=15)
    blocks = _layer_blocks(layer)
    c = 37
    hidden = np.zeros((1, cfg.H), np.uint16)
    hidden[0, c] = 0x3F80   # bf16 1.0
    out = moe.moe_forward(hidden, np.array([[1]], np.int32), np.ones((1, 1), np.float32),
                          blocks, cfg.E)
    codes_gu, luts_gu, q_gu = layer.block(1, 0)
    codes_dn, luts_dn, q_dn = layer.block(1, 1)
    g = np.array([float(luts_gu[q_gu][i, codes_gu[i, c] >> (8 - q_gu)]) for i in range(cfg.I)])
    u = np.array([float(luts_gu[q_gu][cfg.I + i, codes_gu[cfg.I + i, c] >> (8 - q_gu)])
                  for i in range(cfg.I)])
    h = g / (1 + np.exp(-g)) * u
    wd = np.array([[float(luts_dn[q_dn][n, codes_dn[n, i] >> (8 - q_dn)]) for i in range(cfg.I)]
                   for n in range(cfg.H)])
    np.testing.assert_allclose(out[0], wd @ h, rtol=1e-12, atol=1e-18)


# ---------------------------------------------------------------- generator

def test_generator_is_seeded_and_shaped():
    cfg = configs.config_by_name("tiny")
    a = gen.make_layer(cfg, 0)
    b = gen.make_layer(cfg, 0)
    np.testing.assert_array_equal(a.codes_gu, b.codes_gu)
    assert a.codes_gu.shape == (8, 1024, 256) and a.codes_dn.shape == (8, 256, 512)
    for bits in (3, 4, 5, 6, 8):
        assert a.lut_gu[bits].shape == (8, 1024, 1 << bits)
        assert np.all(np.diff(a.lut_gu[bits].astype(np.float32), axis=-1) >= 0)
    assert set(np.unique(a.q)) <= {3, 4, 5, 6, 8}
    t1 = gen.make_tokens(a, 16)
    t2 = gen.make_tokens(b, 16)
    np.testing.assert_array_equal(t1.hidden_bf16, t2.hidden_bf16)


def test_generator_bf16_rounding():
    x = np.array([1.0, -2.5, 1.00390625, 1.01171875, 3.0e-3], np.float32)
    bits = gen.float32_to_bf16_bits(x)
    back = gen.bf16_bits_to_float32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to even (1.0)
    assert back[0] == 1.0 and back[1] == -2.5 and back[2] == 1.0
    assert back[3] == np.float32(1.015625)
    assert abs(back[4] - 3.0e-3) <= 2.0 ** -8 * 3.0e-3   # half an ulp, 8 significant bits


def test_recommit_lowers_one_rung_above_floor():
    cfg = configs.LayerConfig("rc", H=64, I=32, E=32, k=8, T=(4,), q_mode="zipf_floor6",
                              logit_mode="zipf", recommit_frac=0.25)
    layer = gen.make_layer(cfg, 0)
    ids, new_q = gen.make_recommit(layer)
    floor = gen.q_floor(cfg).ravel()
    old = layer.q.ravel()[ids]
    assert len(ids) == 16 and np.all(np.diff(ids) > 0)
    ladder = [3, 4, 5, 6, 8]
    for o, n, f in zip(old, new_q, floor[ids]):
        assert ladder.index(int(n)) == ladder.index(int(o)) - 1 and n >= f


# ---------------------------------------------------------------- planner

def _planner_example():
    return dict(q_now=[8, 6, 8, 4], sensitivity=[1.5, 1, 2, 1], bytes_per_bit=[100] * 4,
                routing_mass=[3, 1], hot_floor=6)


def test_planner_worked_example():
    for target, ids, qs, freed in _read_golden("planner_worked_example.txt"):
        got = planner.plan_recommit(bytes_to_free=int(target), **_planner_example())
        want_ids = [] if ids == "-" else [int(x) for x in ids.split(",")]
        want_q = [] if qs == "-" else [int(x) for x in qs.split(",")]
        assert got == (want_ids, want_q, int(freed)), target


def test_planner_equal_blocks_cut_least_sensitive_first():
    # equal sizes, no hot expert, sensitivities within a factor 6 of each
    # other: every first cut (8 -> 6) is cheaper per byte than any second one,
    # so the first m cuts are the m least sensitive blocks (a stable argsort)
    rng = np.random.default_rng(3)
    n, m = 24, 7
    sens = rng.uniform(1.0, 5.0, n).astype(np.float32)
    ids, qs, freed = planner.plan_recommit([8] * n, sens, [64] * n, [1.0] * (n // 2), 6,
                                           m * 2 * 64)
    assert ids == sorted(np.argsort(sens, kind="stable")[:m].tolist())
    assert qs == [6] * m and freed == m * 2 * 64


def test_planner_invariants_random():
    rng = np.random.default_rng(11)
    for trial in range(20):
        E = int(rng.integers(1, 12))
        n = 2 * E
        q_now = rng.choice(planner.LADDER, n).tolist()
        sens = rng.lognormal(0, 1, n).astype(np.float32)
        bpb = rng.integers(0, 5000, n).tolist()
        mass = rng.exponential(1.0, E).astype(np.float32)
        target = int(rng.integers(0, 60000))
        trace = []
        ids, qs, freed = planner.plan_recommit(q_now, sens, bpb, mass, 6, target, trace)
        total = float(sum(float(m) for m in mass))
        new = list(q_now)
        for i, q in zip(ids, qs):
            new[i] = q
        for i in range(n):
            assert new[i] <= q_now[i]                                   # only lowered
            hot = float(mass[i // 2]) * E > total
            if new[i] != q_now[i]:
                assert new[i] >= (6 if hot else 3)                      # floors respected
        assert freed == sum((q_now[i] - new[i]) * bpb[i] for i in range(n))
        ratios = [r for r, _, _ in trace]
        assert ratios == sorted(ratios)                                 # greedy order
        if freed < target:                                              # nothing left to cut
            assert planner.plan_recommit(new, sens, bpb, mass, 6, 1)[2] == 0
