"""Routed-expert MoE layer over bitplane blocks (oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources:
  * PagedWeight, "Core components" 1: the unit of storage is one linear block
    per (layer, expert, module), the module being gate_up or down; each block
    has its own committed bitwidth q_i in the Weight Page Table.
  * PagedWeight, "Core components" 3 (fused mixed-precision kernel): one fused
    operation reads every block's bitplanes and LUTs at that block's own q_i.

Readings (the pages do not write the layer out):
  * Router: softmax over the E logits (fp64), top-k by a stable descending
    sort (equal probabilities go to the lower expert id), the k kept
    probabilities renormalised to sum to 1.
  * Gate_up block rows 0..I-1 are the gate rows, rows I..2I-1 the up rows;
    h = SiLU(g) * u with SiLU(g) = g / (1 + exp(-g)); y = h W_down^T.
  * Permutation: pair p = t*k + j goes to expert topk_ids[t, j]; pairs are
    grouped by expert, ascending p inside an expert (a stable sort by expert).
  * Combine: out[t] = sum_j topk_weights[t, j] * y_{e_tj}[t], summed in j order.
All floating point here is fp64; bf16 hidden states and fp16 LUT values are
widened exactly.
"""
from typing import Callable, Dict, Optional, Sequence, Tuple

import numpy as np

from .apl import dequant


def bf16_to_float64(bits: np.ndarray) -> np.ndarray:
    """Exact value of raw bf16 bits (the top half of an IEEE float32)."""
    widened = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return widened.view(np.float32).astype(np.float64)


def softmax(logits: np.ndarray) -> np.ndarray:
    z = np.asarray(logits, dtype=np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def route_topk(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k expert ids int32 [T, k] and renormalised weights fp64 [T, k]."""
    p = softmax(logits)
    ids = np.argsort(-p, axis=-1, kind="stable")[:, :k]
    kept = np.take_along_axis(p, ids, axis=-1)
    return ids.astype(np.int32), kept / kept.sum(axis=-1, keepdims=True)


def permute(topk_ids: np.ndarray, E: int):
    """(offsets int32 [E+1], perm int32 [T*k], inv int32 [T*k]).

    perm lists pair ids grouped by expert, ascending within an expert;
    expert e owns perm[offsets[e]:offsets[e+1]]; inv[perm[r]] = r.
    """
    flat = np.asarray(topk_ids, dtype=np.int64).ravel()
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    perm = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return offsets.astype(np.int32), perm.astype(np.int32), inv.astype(np.int32)


def routing_stats(topk_ids: np.ndarray, topk_weights: np.ndarray, E: int):
    """Online routing statistics (PagedWeight, "Core components" 2: an
    expert's routing mass is how often it is selected and with what weight).
    Per expert: the number of (token, j) pairs routed to it and the sum of
    their weights (fp64).  Ids outside [0, E) are left out."""
    ids = np.asarray(topk_ids).ravel()
    w = np.asarray(topk_weights, dtype=np.float64).ravel()
    valid = (ids >= 0) & (ids < E)
    counts = np.bincount(ids[valid], minlength=E).astype(np.int64)
    mass = np.bincount(ids[valid], weights=w[valid], minlength=E)
    return counts, mass


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def expert_mlp(x: np.ndarray, w_gu: np.ndarray, w_dn: np.ndarray) -> np.ndarray:
    """y = (SiLU(x W_gate^T) * (x W_up^T)) W_down^T for x [n, H] (fp64)."""
    I = w_dn.shape[1]
    g = x @ w_gu[:I].T
    u = x @ w_gu[I:].T
    h = silu(g) * u
    return h @ w_dn.T


BlockFn = Callable[[int, int], Tuple[np.ndarray, np.ndarray, int]]


def expert_outputs(hidden_bf16: np.ndarray, topk_ids: np.ndarray, block: BlockFn, E: int,
                   experts: Optional[Sequence[int]] = None,
                   tokens: Optional[Sequence[int]] = None) -> Dict[int, np.ndarray]:
    """y_e(x_t) (fp64 [H]) for every routed pair p = t*k + j, keyed by p.

    block(e, m) returns (planes uint32 [8, K/32, N], lut_q fp16 [N, 2^q], q)
    for block 2e+m (m = 0 gate_up, m = 1 down), as the page table commits it.
    `experts` / `tokens` restrict the pairs computed (default: all).
    """
    x = bf16_to_float64(hidden_bf16)
    T, k = topk_ids.shape
    offsets, perm, _ = permute(topk_ids, E)
    wanted = np.ones(T, bool) if tokens is None else np.isin(np.arange(T), tokens)
    y_pair = {}
    for e in (range(E) if experts is None else experts):
        pairs = [int(p) for p in perm[offsets[e]:offsets[e + 1]] if wanted[p // k]]
        if not pairs:
            continue
        w_gu = dequant(*block(e, 0))
        w_dn = dequant(*block(e, 1))
        y = expert_mlp(x[[p // k for p in pairs]], w_gu, w_dn)
        for r, p in enumerate(pairs):
            y_pair[p] = y[r]
    return y_pair


def combine(y_pair: Dict[int, np.ndarray], topk_weights: np.ndarray, H: int,
            tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """out[t] = sum_j w_tj * y_pair[t*k + j], summed in j order (fp64)."""
    wts = np.asarray(topk_weights, dtype=np.float64)
    T, k = wts.shape
    rows = np.arange(T) if tokens is None else np.asarray(sorted(tokens))
    out = np.zeros((rows.size, H), dtype=np.float64)
    for i, t in enumerate(rows):
        for j in range(k):
            out[i] += wts[t, j] * y_pair[int(t) * k + j]
    return out


def moe_forward(hidden_bf16: np.ndarray, topk_ids: np.ndarray, topk_weights: np.ndarray,
                block: BlockFn, E: int, tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """The layer output, fp64 [T, H] (or [len(tokens), H] for a token subset)."""
    y_pair = expert_outputs(hidden_bf16, topk_ids, block, E, tokens=tokens)
    return combine(y_pair, topk_weights, hidden_bf16.shape[1], tokens=tokens)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    """||got - ref||_2 / ||ref||_2 over the whole tensor (fp64)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))
