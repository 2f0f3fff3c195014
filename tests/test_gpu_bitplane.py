"""Bitplane encoding and top-b read-back on the GPU, bit-exact against the oracle."""
import numpy as np
import pytest

from oracle import apl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pw():
    import any_precision_bitplane_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.lib()
    return m


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("N,K", [(1, 32), (3, 96), (7, 1440), (64, 2048), (2816, 2048),
                                 (33, 32 * 45)])
def test_pack_bit_exact(pw, N, K):
    rng = np.random.default_rng(N * 131 + K)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    planes = pw.pack_bitplanes(torch.from_numpy(codes).cuda())
    np.testing.assert_array_equal(_u32(planes), apl.pack_bitplanes(codes))


@pytest.mark.parametrize("N,K", [(5, 64), (96, 1408), (128, 4096)])
def test_unpack_top_bit_exact(pw, N, K):
    rng = np.random.default_rng(N + K)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    ref_planes = apl.pack_bitplanes(codes)
    planes = torch.from_numpy(ref_planes.view(np.int32)).cuda()
    for b in range(1, 9):
        got = pw.unpack_top(planes, N, K, b).cpu().numpy()
        np.testing.assert_array_equal(got, apl.unpack_top(ref_planes, b))
        np.testing.assert_array_equal(got, codes >> (8 - b))


def test_pack_full_size_block_sampled_rows(pw):
    # Mixtral-sized gate_up block (28672 x 4096): pack on the GPU, compare a
    # sample of rows (incl. first and last) with the oracle's encoding
    N, K = 28672, 4096
    rng = np.random.default_rng(77)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    planes = _u32(pw.pack_bitplanes(torch.from_numpy(codes).cuda()))
    rows = np.concatenate([[0, 1, N - 1], rng.choice(N, 61, replace=False)])
    np.testing.assert_array_equal(planes[:, :, rows], apl.pack_bitplanes(codes[rows]))


def test_pack_worked_example_on_gpu(pw):
    codes = np.zeros((2, 64), np.uint8)
    codes[0, 0], codes[0, 33], codes[1, 31], codes[1, 40] = 176, 1, 255, 66
    planes = _u32(pw.pack_bitplanes(torch.from_numpy(codes).cuda()))
    # planes[p, w, n]: word w of row n
    assert planes[0, 0, 0] == 1 and planes[2, 0, 0] == 1 and planes[3, 0, 0] == 1
    assert planes[7, 1, 0] == 2 and planes[1, 1, 1] == 0x100 and planes[6, 1, 1] == 0x100
    assert all(planes[p, 0, 1] == 0x80000000 for p in range(8))
