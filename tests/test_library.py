"""Host-side checks of libpw: it builds, loads, exports every symbol pw.h
declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pw():
    from any_precision_bitplane_gb300 import build as b
    b.build()
    import any_precision_bitplane_gb300 as m
    m.lib()
    return m


def _header_functions():
    text = open(os.path.join(ROOT, "include", "pw.h")).read()
    return set(re.findall(r"^\s*(?:const char\*|int32_t|int)\s+(pw_\w+)\s*\(", text, re.M))


def test_exports_match_header(pw):
    declared = _header_functions()
    assert declared, "no declarations parsed"
    handle = pw.lib()
    for name in declared:
        assert hasattr(handle, name), name
    assert declared == set(pw.EXPORTED)


def test_version_and_error_string(pw):
    assert pw.lib().pw_version() >= 100
    assert isinstance(pw.last_error(), str)


def test_workspace_bytes(pw):
    n = pw.workspace_bytes(16, 256, 512, 8, 2)
    assert n >= 16 * 2 * 512 * 4 and n % 256 == 0
    assert pw.workspace_bytes(0, 256, 512, 8, 2) >= 0


@pytest.mark.parametrize("shape,code", [
    ((4, 250, 512, 8, 2), 3),   # H not a multiple of 32
    ((4, 256, 500, 8, 2), 3),   # I not a multiple of 32
    ((4, 256, 512, 8, 9), 3),   # k > E
    ((-1, 256, 512, 8, 2), 1),  # negative T
    ((4, 0, 512, 8, 2), 1),
])
def test_shape_validation(pw, shape, code):
    n = ctypes.c_size_t(0)
    s = pw.MoeShape(*shape)
    rc = pw.lib().pw_workspace_bytes(ctypes.byref(s), ctypes.byref(n))
    assert rc == code
    assert pw.last_error()


def test_pack_and_unpack_reject_bad_sizes(pw):
    L = pw.lib()
    assert L.pw_pack_bitplanes(None, 4, 48, None, None) == pw.PW_ERR_SHAPE
    assert L.pw_pack_bitplanes(None, -1, 64, None, None) == pw.PW_ERR_INVALID_ARG
    assert L.pw_unpack_top(None, 4, 64, 9, None, None) == pw.PW_ERR_UNSUPPORTED_Q
    assert L.pw_unpack_top(None, 4, 64, 0, None, None) == pw.PW_ERR_UNSUPPORTED_Q
    # empty work is a no-op, not an error
    assert L.pw_pack_bitplanes(None, 0, 64, None, None) == pw.PW_OK


def test_route_and_permute_limits(pw):
    L = pw.lib()
    assert L.pw_route_topk(None, 4, 2048, 2, None, None, None) == pw.PW_ERR_SHAPE
    assert L.pw_route_topk(None, 4, 8, 9, None, None, None) == pw.PW_ERR_SHAPE
    assert L.pw_route_topk(None, 0, 8, 2, None, None, None) == pw.PW_OK
    assert L.pw_permute(None, 4, 2, 2000, None, None, None, None, None) == pw.PW_ERR_SHAPE


def test_page_table_rejects_bad_entries(pw):
    L = pw.lib()
    arr = (pw.BlockEntry * 2)(pw.BlockEntry(7, 0, 16, 16), pw.BlockEntry(3, 0, 16, 16))
    h = ctypes.c_void_p()
    assert L.pw_page_table_create(2, arr, ctypes.byref(h)) == pw.PW_ERR_UNSUPPORTED_Q
    arr = (pw.BlockEntry * 1)(pw.BlockEntry(3, 5, 16, 16))
    assert L.pw_page_table_create(1, arr, ctypes.byref(h)) == pw.PW_ERR_INVALID_ARG
    arr = (pw.BlockEntry * 1)(pw.BlockEntry(3, 0, 0, 16))
    assert L.pw_page_table_create(1, arr, ctypes.byref(h)) == pw.PW_ERR_INVALID_ARG
    arr = (pw.BlockEntry * 1)(pw.BlockEntry(3, 0, 8, 16))   # misaligned planes
    assert L.pw_page_table_create(1, arr, ctypes.byref(h)) == pw.PW_ERR_INVALID_ARG
    assert L.pw_page_table_create(0, arr, ctypes.byref(h)) == pw.PW_ERR_INVALID_ARG
    assert L.pw_page_table_destroy(None) == pw.PW_OK
    assert L.pw_page_table_commit(None, 1, None, None, None, None) == pw.PW_ERR_INVALID_ARG


def test_forward_rejects_null_table(pw):
    L = pw.lib()
    s = pw.MoeShape(4, 256, 512, 8, 2)
    rc = L.pw_moe_forward(ctypes.byref(s), None, None, None, None, None, None, 0, None)
    assert rc == pw.PW_ERR_INVALID_ARG


# The planner is a host computation inside libpw: it runs without a GPU.

def test_planner_matches_oracle(pw):
    import numpy as np
    from oracle import planner
    rng = np.random.default_rng(5)
    for trial in range(30):
        E = int(rng.integers(1, 40))
        n = 2 * E
        q_now = rng.choice(planner.LADDER, n).astype(np.int32)
        sens = rng.lognormal(0, 1.5, n).astype(np.float32)
        if trial % 3 == 0:
            sens[:] = np.float32(1.0)          # many equal ratios: the tie-break decides
        bpb = rng.integers(0, 1 << 20, n)
        mass = rng.exponential(1.0, E).astype(np.float32)
        target = int(rng.integers(0, int(bpb.sum()) * 3 + 1))
        hot_floor = int(rng.choice(planner.LADDER))
        want = planner.plan_recommit(q_now.tolist(), sens, bpb.tolist(), mass, hot_floor, target)
        got = pw.plan_recommit(q_now, sens, bpb, mass, hot_floor, target)
        assert got == want, trial


def test_planner_rejects_bad_input(pw):
    with pytest.raises(pw.PWError) as ei:
        pw.plan_recommit([8, 7], [1, 1], [10, 10], [1.0], 6, 5)
    assert ei.value.code == pw.PW_ERR_UNSUPPORTED_Q
    with pytest.raises(pw.PWError) as ei:
        pw.plan_recommit([8, 8, 8], [1, 1, 1], [10, 10, 10], [1.0], 6, 5)
    assert ei.value.code == pw.PW_ERR_INVALID_ARG
    assert pw.plan_recommit([], [], [], [], 6, 5) == ([], [], 0)
