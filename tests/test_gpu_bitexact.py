"""Bit-exact checks of the index, lookup, grouping and gather work the kernels
do, against the oracle (PagedWeight, "Core components" 1: a b-bit view reads
the top b planes, idx = code >> (8 - b), and the weight is the row's LUT
entry; "Core components" 3: one fused operation over the routed pairs).

The index and lookup checks run the forward kernels' own device code (the
decode kernels' nibble and byte extraction and their pair / fp32 tables, the
tensor-core dequant warps' half-word extraction and fp16 LUT layout) on whole
blocks at the Qwen1.5-shaped sizes and on ragged ones.  The grouping and the
gathered activations are read back from a forward call's workspace.  Every
comparison is exact."""
import numpy as np
import pytest

from oracle import apl, moe
from workloads import configs, gen
from helpers import host_layer, oracle_route

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

QS = (3, 4, 5, 6, 8)
# (N, K): Qwen1.5-shaped gate_up and down blocks, a ragged pair, the smallest
BLOCKS = [(2816, 2048), (2048, 1408), (96, 96), (32, 32)]


@pytest.fixture(scope="module")
def pw():
    import any_precision_bitplane_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.lib()
    return m


def _block(N, K, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    planes = apl.pack_bitplanes(codes)
    return codes, planes, torch.from_numpy(planes.view(np.int32)).cuda()


@pytest.mark.parametrize("N,K", BLOCKS)
def test_index_forms_match_unpack_top(pw, N, K):
    codes, planes, d_planes = _block(N, K, seed=N + K)
    for q in QS:
        want = apl.unpack_top(planes, q)
        forms = [pw.INDEX_BYTES, pw.INDEX_HALVES] + ([pw.INDEX_NIBBLES] if q <= 4 else [])
        for form in forms:
            got = pw.debug_index(d_planes, N, K, q, form).cpu().numpy()
            assert np.array_equal(got, want), (q, form)
        assert np.array_equal(want, codes >> (8 - q))


@pytest.mark.parametrize("N,K", BLOCKS)
def test_table_lookups_match_dequant(pw, N, K):
    codes, planes, d_planes = _block(N, K, seed=3 * N + K)
    rng = np.random.default_rng(N)
    for q in QS:
        lut = np.sort(rng.normal(0, 0.02, (N, 1 << q)).astype(np.float16), axis=1)
        want = apl.dequant(planes, lut, q)                     # fp64 of the fp16 entries
        d_lut = torch.from_numpy(lut.view(np.int16)).cuda()
        for path in (pw.PATH_DECODE, pw.PATH_PREFILL):
            got = pw.debug_dequant(d_planes, d_lut, N, K, q, path).cpu().numpy()
            assert np.array_equal(got.astype(np.float64), want), (q, path)


def _positions_fp32(c):
    return 4 * (c % 8) + c // 8          # the fp32 form's order inside a group of 32


def _positions_fp16(c):
    return 8 * (c % 4) + 2 * (c // 8) + (c // 4) % 2   # the fp16 records' order


def _read(ws, off, n, dtype):
    return ws[off:off + n].cpu().numpy().view(dtype)


@pytest.mark.parametrize("name,T", [("qwen15_decode", 8), ("qwen3_decode", 64), ("tiny", 16)])
def test_decode_grouping_and_activation_forms(pw, name, T):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = host_layer(name)
    cfg = layer.cfg
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, cfg.k)
        ws = torch.zeros(pw.workspace_bytes(T, cfg.H, cfg.I, cfg.E, cfg.k), dtype=torch.uint8,
                         device="cuda")
        pw.moe_forward(torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
                       torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), dl.table, cfg.I,
                       cfg.E, workspace=ws, path=pw.PATH_DECODE)
        torch.cuda.synchronize()
        sec = [pw.debug_workspace_section(T, cfg.H, cfg.I, cfg.E, cfg.k, pw.PATH_DECODE, i)
               for i in range(4)]
        offsets = _read(ws, *sec[0], np.int32)
        perm = _read(ws, *sec[1], np.int32)
        xs = _read(ws, *sec[2], np.float32).reshape(T, cfg.H // 32, 32)
        rec = ws[sec[3][0]:sec[3][0] + sec[3][1]].cpu().numpy().reshape(T, cfg.H // 32, 80)
    finally:
        dl.close()
    want_off, want_perm, _ = moe.permute(ids, cfg.E)
    assert np.array_equal(offsets, want_off)
    assert np.array_equal(perm, want_perm)
    x = gen.bf16_bits_to_float32(tok.hidden_bf16).reshape(T, cfg.H // 32, 32)
    cols = np.arange(32)
    # fp32 form: every hidden value, exactly, at its position
    assert np.array_equal(xs[:, :, _positions_fp32(cols)], x)
    # fp16 records: the scale of each half of a group is 2^e with e the
    # exponent of the half's largest magnitude (from the oracle's values), and
    # each value is fp16(x * 2^-e) of its own column, exactly
    vals = rec[:, :, :64].copy().view(np.float16)[:, :, _positions_fp16(cols)]
    scales = rec[:, :, 64:72].copy().view(np.float32).astype(np.float64)   # [T, G, 2]
    xh = x.astype(np.float64).reshape(T, cfg.H // 32, 2, 16)
    _, ex = np.frexp(np.abs(xh).max(axis=3))                                # max = m 2^ex, m in [0.5, 1)
    want_scale = np.where(np.abs(xh).max(axis=3) > 0, np.ldexp(1.0, ex - 1), np.ldexp(1.0, -126))
    assert np.array_equal(scales, want_scale)
    want_vals = (xh / want_scale[..., None]).astype(np.float16).reshape(T, cfg.H // 32, 32)
    assert np.array_equal(vals.view(np.uint16), want_vals.view(np.uint16))


@pytest.mark.parametrize("spec", [("g_small", 256, 128, 4, 2, 300), ("g_many", 256, 64, 16, 4, 257)],
                         ids=["g_small", "g_many"])
def test_prefill_grouping_and_gathered_rows(pw, spec):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    name, H, I, E, k, T = spec
    layer = gen.make_layer(configs.custom(name, H, I, E, k, T), seed=33)
    dl = DeviceLayer(layer)
    try:
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, k)
        ws = torch.zeros(pw.workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device="cuda")
        pw.moe_forward(torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
                       torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), dl.table, I, E,
                       workspace=ws, path=pw.PATH_PREFILL)
        torch.cuda.synchronize()
        sec = [pw.debug_workspace_section(T, H, I, E, k, pw.PATH_PREFILL, i) for i in range(4)]
        offsets = _read(ws, *sec[0], np.int32)
        perm = _read(ws, *sec[1], np.int32)
        xg = _read(ws, *sec[2], np.float16).reshape(T * k, H).astype(np.float64)
        scale = _read(ws, *sec[3], np.float32).astype(np.float64)
    finally:
        dl.close()
    want_off, want_perm, _ = moe.permute(ids, E)
    assert np.array_equal(offsets, want_off)
    assert np.array_equal(perm, want_perm)
    x = gen.bf16_bits_to_float32(tok.hidden_bf16).astype(np.float64)
    # gathered row r is fp16(hidden row of pair perm[r] * 2^-e), exactly, with
    # 2^e (the row's scale) from the exponent of the row's largest magnitude
    rows = x[perm // k]
    rmax = np.abs(rows).max(axis=1)
    _, ex = np.frexp(rmax)
    want_scale = np.where(rmax > 0, np.ldexp(1.0, ex - 1), np.ldexp(1.0, -126))
    assert np.array_equal(scale, want_scale)
    want = (rows / want_scale[:, None]).astype(np.float16).astype(np.float64)
    assert np.array_equal(xg, want)
