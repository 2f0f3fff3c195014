"""Activations far outside fp16's range, on every path of the fused layer.

The tensor-core path stores its fp16 operands with a power-of-two scale per
gathered row (and h with the square of it); the decode kernels keep fp32
activations, or fp16 records with a power-of-two scale per 16 columns.  So a
hidden row of magnitude 2^40 or 2^-30 must give the oracle's output to the
usual tolerance, token by token (the rows differ by 2^70, so one pooled norm
would only see the largest)."""
import numpy as np
import pytest

from helpers import REL_TOL, oracle_out, oracle_route
from workloads import configs, gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# exponent shifts applied to whole hidden rows (exact in bf16)
SHIFTS = (40, -30, 10, -10, 0)


@pytest.fixture(scope="module")
def pw():
    import any_precision_bitplane_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.lib()
    return m


def _scaled_tokens(layer, T):
    tok = gen.make_tokens(layer, T)
    x = gen.bf16_bits_to_float32(tok.hidden_bf16).astype(np.float64)
    for t in range(T):
        x[t] *= 2.0 ** SHIFTS[t % len(SHIFTS)]
    bits = gen.float32_to_bf16_bits(x.astype(np.float32))
    # a power-of-two scaling of a bf16 value is exact
    assert np.array_equal(gen.bf16_bits_to_float32(bits).astype(np.float64), x)
    return gen.Tokens(bits, tok.logits)


@pytest.mark.parametrize("case", ["prefill", "decode_hybrid", "decode_small"])
def test_large_and_small_activations(pw, case):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    # H, I suit the tensor-core kernels (H % 128, I % 64); 32 tokens over 4
    # experts put ~16 pairs on each, so the decode call sends them to the
    # GEMM kernels (the hybrid path); 5 tokens stay on the decode kernels
    T = 5 if case == "decode_small" else 32
    layer = gen.make_layer(configs.custom("range", 256, 128, 4, 2, T), seed=41)
    dl = DeviceLayer(layer)
    try:
        tok = _scaled_tokens(layer, T)
        ids, w = oracle_route(tok, 2)
        path = pw.PATH_PREFILL if case == "prefill" else pw.PATH_DECODE
        out = pw.moe_forward(torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
                             torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                             dl.table, dl.I, dl.E, path=path).cpu().numpy()
        assert dl.table.status() == pw.PW_OK
    finally:
        dl.close()
    ref = oracle_out(layer, tok.hidden_bf16, ids, w)
    assert np.isfinite(out).all()
    per_token = np.linalg.norm(out - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert per_token.max() <= REL_TOL, (int(per_token.argmax()), float(per_token.max()))
