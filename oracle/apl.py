"""Overlay bitplane format with per-row lookup tables (oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: PagedWeight, "Core components" 1 (Paged Weight representation): the
weights are held in Any-Precision's overlay bitplane format with associated
lookup tables; a b-bit view of a block reads its top b bitplanes.

Readings (the pages give no layout):
  * n = 8 planes per block; plane p holds bit (7 - p) of every 8-bit code, so
    plane 0 is the most significant and the top-b planes are planes 0..b-1,
    a contiguous prefix of the storage.
  * Plane-major, word-major layout uint32 [8][K/32][N]: plane p's word w of
    row n holds weights k = 32w .. 32w+31 of that row, weight k at bit
    (k mod 32) (LSB first); the N words of one word column are contiguous.
  * Reading the top b planes gives idx_b = sum_{p<b} bit_p << (b-1-p), which
    equals code >> (8 - b).
  * Row n's b-bit lookup table holds 2^b fp16 values; the weight is
    LUT_q[n][idx_q] at the block's committed bitwidth q.
"""
import numpy as np

PLANES = 8


def pack_bitplanes(codes: np.ndarray) -> np.ndarray:
    """Encode 8-bit codes [N, K] as 8 bitplanes, uint32 [8, K/32, N].

    np.packbits with little bit order puts column 32w+t at bit t of word w
    once the bytes are read as little-endian uint32.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    N, K = codes.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    planes = np.empty((PLANES, K // 32, N), dtype=np.uint32)
    for p in range(PLANES):
        bit = (codes >> (7 - p)) & 1                            # plane p = bit (7-p)
        packed = np.packbits(bit, axis=1, bitorder="little")    # [N, K/8] bytes
        planes[p] = np.ascontiguousarray(packed).view("<u4").T  # words [N, K/32] -> [K/32, N]
    return planes


def unpack_top(planes: np.ndarray, b: int) -> np.ndarray:
    """Read the top b planes back into b-bit indices, uint8 [N, K]."""
    planes = np.asarray(planes, dtype=np.uint32)
    if not 1 <= b <= planes.shape[0]:
        raise ValueError("b out of range")
    _, W, N = planes.shape
    idx = np.zeros((N, W * 32), dtype=np.uint8)
    for p in range(b):
        as_bytes = np.ascontiguousarray(planes[p].T).astype("<u4").view(np.uint8)
        plane_bit = np.unpackbits(as_bytes, axis=1, bitorder="little")  # column k = bit k%32 of word k/32
        idx = (idx << 1) | plane_bit        # plane 0 ends up as the top index bit
    return idx


def dequant(planes: np.ndarray, lut_q: np.ndarray, q: int) -> np.ndarray:
    """Weights of a block at committed bitwidth q: W[n,k] = LUT_q[n][idx_q[n,k]] (fp64)."""
    lut_q = np.asarray(lut_q)
    if lut_q.shape[-1] != (1 << q):
        raise ValueError("LUT width must be 2^q")
    idx = unpack_top(planes, q)
    rows = np.arange(idx.shape[0])[:, None]
    return lut_q[rows, idx].astype(np.float64)
