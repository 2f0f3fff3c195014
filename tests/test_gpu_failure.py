"""Failure detection on the device: every wait of the forward kernels is
bounded, and one that runs out latches PW_ERR_TIMEOUT and returns.

The waits run against something nothing releases (a counter nobody
increments, an mbarrier phase that never completes), with a short limit, so
no GPU hangs or faults; afterwards the context must still run a forward call
that matches the oracle."""
import time

import numpy as np
import pytest

from helpers import REL_TOL, host_layer, oracle_out, oracle_route, rel_l2
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


@pytest.fixture(scope="module")
def dl(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    d = DeviceLayer(host_layer("tiny"))
    yield d
    d.close()


@pytest.mark.parametrize("which,polls", [(0, 2000), (1, 64)], ids=["gate_up_counter", "mbarrier"])
def test_bounded_wait_runs_out_and_latches_timeout(pw, dl, which, polls):
    assert dl.table.status(reset=True) == pw.PW_OK
    t0 = time.perf_counter()
    pw.debug_bounded_wait(dl.table, which, polls)
    status = dl.table.status(reset=True)          # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == pw.PW_ERR_TIMEOUT
    assert elapsed < 30.0


def test_context_usable_after_timeouts(pw, dl):
    for which, polls in ((0, 500), (1, 16)):
        pw.debug_bounded_wait(dl.table, which, polls)
    assert dl.table.status(reset=True) == pw.PW_ERR_TIMEOUT
    layer = host_layer("tiny")
    tok = gen.make_tokens(layer, 16)
    ids, w = oracle_route(tok, layer.cfg.k)
    out = pw.moe_forward(torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
                         torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                         dl.table, dl.I, dl.E)
    assert dl.table.status() == pw.PW_OK
    assert rel_l2(out.cpu().numpy(), oracle_out(layer, tok.hidden_bf16, ids, w)) <= REL_TOL


def test_bounded_wait_rejects_bad_arguments(pw, dl):
    for which, polls in ((2, 10), (0, 0), (1, (1 << 20) + 1)):
        with pytest.raises(pw.PWError) as ei:
            pw.debug_bounded_wait(dl.table, which, polls)
        assert ei.value.code == pw.PW_ERR_INVALID_ARG


def test_traces_need_the_traced_build(pw):
    # libpw.so is built without the GEMM and decode traces: the readers say
    # so and change nothing (a traced library, build.py --trace, fills them)
    with pytest.raises(pw.PWError) as e:
        pw.debug_gemm_trace()
    assert e.value.code == pw.PW_ERR_NOT_BUILT
    with pytest.raises(pw.PWError) as e:
        pw.debug_decode_trace()
    assert e.value.code == pw.PW_ERR_NOT_BUILT
