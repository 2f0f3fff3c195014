"""The decode trace summary (trace_decode.summarize) on a hand-built record:
per-bitwidth medians, phase shares and the tail's idle times worked out by
hand."""
import numpy as np
import pytest

from any_precision_bitplane_gb300 import trace_decode


def _record():
    tile = np.zeros((16, 32, 10), np.uint64)
    cta = np.zeros((16, 2), np.uint64)
    # fields: start ns, end ns, descriptor, set-up, columns, reduction,
    # q + 256 * pairs, set-up parts (issue, LUT wait + build, barrier)
    tile[0, 0] = [1000, 11000, 100, 400, 1000, 200, 4 + 256 * 1, 100, 250, 50]
    tile[0, 1] = [12000, 20000, 300, 600, 2000, 100, 8 + 256 * 2, 200, 350, 50]
    tile[2, 0] = [1500, 9500, 200, 500, 1500, 300, 4 + 256 * 1, 150, 300, 50]
    cta[0] = [5 + 1, 21000]    # CTA 0 on SM 5, exits at 21 us
    cta[2] = [7 + 1, 10000]    # CTA 38 on SM 7, exits at 10 us
    return tile, cta


def test_per_bitwidth_medians():
    sm = trace_decode.summarize(*_record())
    q4, q8 = sm["per_q"][4], sm["per_q"][8]
    assert q4["tiles"] == 2 and q8["tiles"] == 1
    assert q4["phases"] == [150.0, 450.0, 1250.0, 250.0]
    assert q4["setup_parts"] == [125.0, 275.0, 50.0]
    assert q4["pairs"] == 1.0 and q4["tile_us"] == pytest.approx(9.0)
    assert q8["phases"] == [300.0, 600.0, 2000.0, 100.0]
    assert q8["pairs"] == 2.0 and q8["tile_us"] == pytest.approx(8.0)


def test_all_tiles_and_shares():
    a = trace_decode.summarize(*_record())["all"]
    assert a["tiles"] == 3
    assert a["phases"] == [200.0, 500.0, 1500.0, 200.0]
    assert a["shares"] == pytest.approx([200 / 2400, 500 / 2400, 1500 / 2400, 200 / 2400])


def test_tail_of_the_traced_ctas():
    sm = trace_decode.summarize(*_record())
    assert sm["span_us"] == pytest.approx(20.0)
    (c0, sm0, n0, ex0, idle0), (c1, sm1, n1, ex1, idle1) = sm["ctas"]
    assert (c0, sm0, n0) == (0, 5, 2) and (c1, sm1, n1) == (38, 7, 1)
    assert ex0 == pytest.approx(20.0) and idle0 == pytest.approx(0.0)
    assert ex1 == pytest.approx(9.0) and idle1 == pytest.approx(11.0)


# ---- the tensor-core GEMM trace (trace_gemm.summarize)

from any_precision_bitplane_gb300 import trace_gemm  # noqa: E402


def _gemm_record():
    step = np.zeros((16, 256, 4), np.uint64)
    tile = np.zeros((16, 32, 6), np.uint64)
    smid = np.zeros(16, np.uint64)
    # CTA 0 (trace slot 0) on SM 3: tile 0 issues k-steps 0-3 every 450 ns;
    # tile 1 starts after the epilogue with k-steps 4-5
    issued = [1000, 1450, 1900, 2350, 9000, 9450]
    for i, t in enumerate(issued):
        found = t - 100
        step[0, i] = [found, t, found - 128, t - 500]   # found full, issued, announced, empty
    tile[0, 0] = [900, 2400, 2500, 8800, 100, 800]      # mma, commit, epi start/end, lut
    tile[0, 1] = [8900, 9600, 0, 0, 8100, 8800]
    smid[0] = 3 + 1
    return step, tile, smid


def test_gemm_intervals_of_one_cta():
    per_cta, _ = trace_gemm.summarize(*_gemm_record())
    (cta, sm, iv), = per_cta
    assert (cta, sm, iv["tiles"]) == (0, 3, 2)
    assert iv["kstep"] == [450, 450, 450, 450]      # the 6650 ns tile-boundary gap is dropped
    assert iv["slack"] == [128] * 6
    assert iv["mma"] == [1500, 700]
    assert iv["epi"] == [6300]                      # tile 1's epilogue not reached
    assert iv["idle"] == [6500]                     # last commit 2400 -> next MMA start 8900
    assert iv["lut"] == [700, 700]


def test_gemm_medians_over_ctas():
    step, tile, smid = _gemm_record()
    # a second traced CTA (slot 3, CTA 30) with a slower k-step
    for i, t in enumerate([500, 1100, 1700]):
        step[3, i] = [t - 50, t, t - 90, t - 300]
    tile[3, 0] = [400, 1800, 1900, 5000, 10, 510]
    smid[3] = 9 + 1
    per_cta, med = trace_gemm.summarize(step, tile, smid)
    assert [c for c, _, _ in per_cta] == [0, 30]
    assert med["kstep"] == pytest.approx(450.0)     # median of 450 x4 and 600 x2
    assert med["slack"] == pytest.approx(128.0)     # median of 128 x6 and 40 x3
    assert med["mma"] == pytest.approx(1400.0)      # median of 1500, 700, 1400
    assert med["idle"] == pytest.approx(6500.0)
