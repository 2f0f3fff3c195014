"""Page movement: tail planes offloaded to pinned host memory and reloaded on a
side stream, with the bitwidth raise committed after the reload's event; a
whole block moved out (not resident) and back to new device pages.  Copies are
checked byte for byte, forward calls against the oracle."""
import numpy as np
import pytest

from helpers import REL_TOL, oracle_out, oracle_route, rel_l2
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


@pytest.fixture()
def setup(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = gen.make_layer(configs.custom("pages", 256, 128, 4, 2, 12), seed=71)
    dl = DeviceLayer(layer)
    tok = gen.make_tokens(layer, 12)
    ids, w = oracle_route(tok, 2)
    args = (torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
            torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    yield layer, dl, tok, ids, w, args
    dl.close()


def _fwd(pw, dl, args, stream=None):
    with torch.cuda.stream(stream or torch.cuda.current_stream()):
        return pw.moe_forward(*args, dl.table, dl.I, dl.E)


def test_tail_offload_and_reload_with_commit_after(pw, setup):
    layer, dl, tok, ids, w, args = setup
    e = int(ids[0, 0])
    b = 2 * e                          # the gate_up block of a routed expert: N = 2I, K = H
    N, K = 2 * dl.I, dl.H
    planes = dl.planes_gu[e]
    keep = 3
    dl.commit([b], [keep])
    host = torch.empty((8 - keep) * N * K // 8, dtype=torch.uint8).pin_memory()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    pw.planes_to_host(planes, N, K, keep, host, stream=side)
    side.synchronize()
    want = planes[keep:].contiguous().view(torch.uint8).cpu().reshape(-1)
    assert torch.equal(host, want)
    planes[keep:].fill_(0)             # the tail's device memory is reused
    got = _fwd(pw, dl, args).cpu().numpy()
    assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w, q=dl.q)) <= REL_TOL
    # reload on the side stream; raise the bitwidth only after it has landed
    side.wait_stream(torch.cuda.current_stream())
    pw.planes_from_host(host, planes, N, K, keep, stream=side)
    ready = torch.cuda.Event()
    ready.record(side)
    dl.table.commit_after([b], [8], [dl.lut_ptr(b, 8)], ready)
    dl.q[e, 0] = 8
    got = _fwd(pw, dl, args).cpu().numpy()
    assert dl.table.status() == pw.PW_OK
    assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w, q=dl.q)) <= REL_TOL


def test_whole_block_out_and_back_to_new_pages(pw, setup):
    layer, dl, tok, ids, w, args = setup
    e = int(ids[0, 0])
    b = 2 * e + 1                      # the down block: N = H, K = I
    N, K = dl.H, dl.I
    ref = _fwd(pw, dl, args).cpu().numpy()
    host = torch.empty(8 * N * K // 8, dtype=torch.uint8).pin_memory()
    pw.planes_to_host(dl.planes_dn[e], N, K, 0, host)
    dl.table.set_pages([b], [dl.planes_ptr(b)], [pw.PW_PAGE_CPU])
    torch.cuda.synchronize()
    got = _fwd(pw, dl, args).cpu().numpy()
    assert dl.table.status() == pw.PW_ERR_PAGE_NOT_RESIDENT
    assert rel_l2(got, oracle_out(layer, tok.hidden_bf16, ids, w, q=dl.q,
                                  drop_experts=[e])) <= REL_TOL
    fresh = torch.empty_like(dl.planes_dn[e])
    side = torch.cuda.Stream()
    pw.planes_from_host(host, fresh, N, K, 0, stream=side)
    ready = torch.cuda.Event()
    ready.record(side)
    torch.cuda.current_stream().wait_event(ready)
    dl.table.set_pages([b], [fresh.data_ptr()], [pw.PW_PAGE_GPU])
    got = _fwd(pw, dl, args).cpu().numpy()
    assert dl.table.status() == pw.PW_OK
    np.testing.assert_array_equal(got, ref)        # same bytes, same result
    dl.table.set_pages([b], [dl.planes_ptr(b)], [pw.PW_PAGE_GPU])
    torch.cuda.synchronize()


def test_page_copy_rejects_bad_arguments(pw, setup):
    layer, dl, *_ = setup
    host = torch.empty(16, dtype=torch.uint8).pin_memory()
    with pytest.raises(pw.PWError) as ei:
        pw.planes_to_host(dl.planes_gu[0], 2 * dl.I, 33, 0, host)
    assert ei.value.code == pw.PW_ERR_SHAPE
    with pytest.raises(pw.PWError) as ei:
        pw.planes_to_host(dl.planes_gu[0], 2 * dl.I, dl.H, 8, host)
    assert ei.value.code == pw.PW_ERR_INVALID_ARG
