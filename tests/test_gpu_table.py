"""Weight Page Table on the GPU: recommits at a safe boundary, CUDA-graph replay
across a commit, page relocation and the device-side status word."""
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


ZIPF = configs.LayerConfig("zipf_small", H=256, I=128, E=32, k=8, T=(64,),
                           q_mode="zipf_floor6", logit_mode="zipf", recommit_frac=0.25)


@pytest.fixture(scope="module")
def setup(pw):
    from any_precision_bitplane_gb300.layer import DeviceLayer
    layer = gen.make_layer(ZIPF, 0)
    dl = DeviceLayer(layer)
    tok = gen.make_tokens(layer, 64)
    ids, w = oracle_route(tok, ZIPF.k)
    args = (torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda(),
            torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    yield layer, dl, tok, ids, w, args
    dl.close()


def _fwd(pw, dl, args, out=None, ws=None):
    return pw.moe_forward(*args, dl.table, dl.I, dl.E, out=out, workspace=ws)


def test_recommit_takes_effect_between_steps(pw, setup):
    layer, dl, tok, ids, w, args = setup
    q_old = dl.q.copy()
    before = _fwd(pw, dl, args).cpu().numpy()
    blocks, new_q = gen.make_recommit(layer)
    assert len(blocks) == 16
    dl.commit(blocks, new_q)
    after = _fwd(pw, dl, args).cpu().numpy()
    q_new = dl.q.copy()
    assert not np.array_equal(q_old, q_new)
    assert rel_l2(before, oracle_out(layer, tok.hidden_bf16, ids, w, q=q_old)) <= REL_TOL
    assert rel_l2(after, oracle_out(layer, tok.hidden_bf16, ids, w, q=q_new)) <= REL_TOL
    entries = dl.table.read()
    for b, q in zip(blocks, new_q):
        assert entries[b][0] == q and entries[b][3] == dl.lut_ptr(b, q)
    # restore the drawn bitwidths for the other tests
    dl.commit(list(range(2 * ZIPF.E)), q_old.ravel().tolist())
    assert dl.table.status() == pw.PW_OK


def test_graph_replay_sees_commit(pw, setup):
    layer, dl, tok, ids, w, args = setup
    q_old = dl.q.copy()
    T, H = args[0].shape
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(pw.workspace_bytes(T, H, dl.I, dl.E, ZIPF.k), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _fwd(pw, dl, args, out, ws)          # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _fwd(pw, dl, args, out, ws)
    g.replay()
    torch.cuda.synchronize()
    r_old = out.cpu().numpy().copy()
    blocks, new_q = gen.make_recommit(layer)
    dl.commit(blocks, new_q)
    g.replay()
    torch.cuda.synchronize()
    r_new = out.cpu().numpy().copy()
    assert rel_l2(r_old, oracle_out(layer, tok.hidden_bf16, ids, w, q=q_old)) <= REL_TOL
    assert rel_l2(r_new, oracle_out(layer, tok.hidden_bf16, ids, w, q=dl.q)) <= REL_TOL
    dl.commit(list(range(2 * ZIPF.E)), q_old.ravel().tolist())
    torch.cuda.synchronize()


def test_page_relocation_is_bit_identical(pw, setup):
    # only the mapping changes: the output must not change by a single bit
    layer, dl, tok, ids, w, args = setup
    ref = _fwd(pw, dl, args).cpu().numpy()
    routed = sorted(set(int(e) for e in np.unique(ids)))
    blocks = [2 * e + m for e in routed[:6] for m in (0, 1)]
    copies = [(dl.planes_gu if b % 2 == 0 else dl.planes_dn)[b // 2].clone() for b in blocks]
    dl.table.set_pages(blocks, [c.data_ptr() for c in copies], [pw.PW_PAGE_GPU] * len(blocks))
    # scribble over the old pages: a stale read would show up
    for b in blocks:
        (dl.planes_gu if b % 2 == 0 else dl.planes_dn)[b // 2].fill_(-1)
    moved = _fwd(pw, dl, args).cpu().numpy()
    torch.cuda.synchronize()
    for b, c in zip(blocks, copies):
        (dl.planes_gu if b % 2 == 0 else dl.planes_dn)[b // 2].copy_(c)
    dl.table.set_pages(blocks, [dl.planes_ptr(b) for b in blocks], [pw.PW_PAGE_GPU] * len(blocks))
    back = _fwd(pw, dl, args).cpu().numpy()
    np.testing.assert_array_equal(moved, ref)
    np.testing.assert_array_equal(back, ref)
    assert dl.table.status() == pw.PW_OK


def test_non_resident_page_is_skipped_and_reported(pw, setup):
    layer, dl, tok, ids, w, args = setup
    e = int(ids[0, 0])
    dl.table.set_pages([2 * e + 1], [dl.planes_ptr(2 * e + 1)], [pw.PW_PAGE_CPU])
    got = _fwd(pw, dl, args).cpu().numpy()
    assert dl.table.status() == pw.PW_ERR_PAGE_NOT_RESIDENT
    ref = oracle_out(layer, tok.hidden_bf16, ids, w, q=dl.q, drop_experts=[e])
    assert rel_l2(got, ref) <= REL_TOL
    dl.table.set_pages([2 * e + 1], [dl.planes_ptr(2 * e + 1)], [pw.PW_PAGE_GPU])
    _fwd(pw, dl, args)
    assert dl.table.status() == pw.PW_OK


def test_bad_expert_id_is_skipped_and_reported(pw, setup):
    layer, dl, tok, ids, w, args = setup
    bad = ids.copy()
    bad[3, 1] = ZIPF.E + 5
    bad[7, 0] = -2
    got = pw.moe_forward(args[0], torch.from_numpy(bad).cuda(), args[2], dl.table, dl.I,
                         dl.E).cpu().numpy()
    assert dl.table.status() == pw.PW_ERR_BAD_EXPERT_ID
    fixed, w0 = ids.copy(), w.copy()
    w0[3, 1] = 0.0
    w0[7, 0] = 0.0
    ref = oracle_out(layer, tok.hidden_bf16, fixed, w0, q=dl.q)
    assert rel_l2(got, ref) <= REL_TOL


def test_commit_rejects_bad_requests(pw, setup):
    layer, dl, *_ = setup
    with pytest.raises(pw.PWError) as ei:
        dl.table.commit([0], [7], [dl.lut_ptr(0, 8)])
    assert ei.value.code == pw.PW_ERR_UNSUPPORTED_Q
    with pytest.raises(pw.PWError) as ei:
        dl.table.commit([2 * ZIPF.E], [3], [dl.lut_ptr(0, 3)])
    assert ei.value.code == pw.PW_ERR_INVALID_ARG
