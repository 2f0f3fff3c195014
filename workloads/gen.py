"""Seeded generator for the synthetic MoE-layer inputs.

Recipe (one numpy.random.default_rng(seed) stream per layer, fixed draw order):
  1. 8-bit weight codes, uniform on [0, 255]: gate_up codes [E, 2I, H], then
     down codes [E, H, I].  Rows 0..I-1 of gate_up are the gate rows and rows
     I..2I-1 the up rows.
  2. Per-row lookup tables: for b in (3, 4, 5, 6, 8), 2^b values per row drawn
     from N(0, 0.02), rounded to fp16 and sorted ascending; gate_up tables
     [E, 2I, 2^b] then down tables [E, H, 2^b].  Tables for different b are
     drawn independently.
  3. Committed bitwidth q per block [E, 2] (column 0 gate_up, column 1 down).
  4. Per token count T, from a copy of the stream state after step 3:
     hidden states N(0, 1) rounded to bf16 (kept as raw uint16 bits), then
     router logits [T, E] (float32).

Nothing here encodes, decodes, routes or multiplies: those steps belong to the
layer and live in the oracle and in the CUDA library.
"""
from dataclasses import dataclass
from typing import Dict, Tuple

import numpy as np

from .configs import BITWIDTHS, LayerConfig


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); return raw uint16 bits."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((bits >> 16) & 1) + np.uint32(0x7FFF)
    return ((bits + bias) >> 16).astype(np.uint16)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def expert_popularity(cfg: LayerConfig) -> np.ndarray:
    """Zipf popularity p_e proportional to (e+1)^-s, normalised (expert-id order)."""
    ranks = np.arange(1, cfg.E + 1, dtype=np.float64)
    p = ranks ** (-cfg.zipf_s)
    return p / p.sum()


def q_floor(cfg: LayerConfig) -> np.ndarray:
    """Lowest bitwidth each block may be committed to, [E, 2]."""
    floor = np.full((cfg.E, 2), BITWIDTHS[0], dtype=np.int32)
    if cfg.q_mode == "zipf_floor6":
        hot = expert_popularity(cfg) > 1.0 / cfg.E
        floor[hot] = 6
    elif cfg.q_mode == "hot8_rest34":
        floor[list(cfg.hot)] = 8
    return floor


@dataclass
class Layer:
    cfg: LayerConfig
    codes_gu: np.ndarray            # uint8 [E, 2I, H]
    codes_dn: np.ndarray            # uint8 [E, H, I]
    lut_gu: Dict[int, np.ndarray]   # b -> float16 [E, 2I, 2^b]
    lut_dn: Dict[int, np.ndarray]   # b -> float16 [E, H, 2^b]
    q: np.ndarray                   # int32 [E, 2]
    rng_state: dict                 # stream state after the weights were drawn

    def block(self, e: int, m: int):
        """(codes [N, K], {b: lut [N, 2^b]}, q) of block 2e+m."""
        if m == 0:
            return self.codes_gu[e], {b: t[e] for b, t in self.lut_gu.items()}, int(self.q[e, 0])
        return self.codes_dn[e], {b: t[e] for b, t in self.lut_dn.items()}, int(self.q[e, 1])


@dataclass
class Tokens:
    hidden_bf16: np.ndarray   # uint16 [T, H] raw bf16 bits
    logits: np.ndarray        # float32 [T, E]


def _draw_luts(rng, E: int, N: int, b: int) -> np.ndarray:
    vals = rng.normal(0.0, 0.02, size=(E, N, 1 << b)).astype(np.float16)
    vals.sort(axis=-1)
    return vals


def _draw_q(rng, cfg: LayerConfig) -> np.ndarray:
    choices = np.asarray(BITWIDTHS, dtype=np.int32)
    if cfg.q_mode == "uniform":
        return rng.choice(choices, size=(cfg.E, 2)).astype(np.int32)
    if cfg.q_mode == "hot8_rest34":
        q = rng.choice(np.asarray((3, 4), np.int32), size=(cfg.E, 2)).astype(np.int32)
        q[list(cfg.hot)] = 8
        return q
    if cfg.q_mode == "zipf_floor6":
        q = rng.choice(choices, size=(cfg.E, 2)).astype(np.int32)
        return np.maximum(q, q_floor(cfg))
    raise ValueError(cfg.q_mode)


def make_layer(cfg: LayerConfig, seed: int = 0) -> Layer:
    rng = np.random.default_rng(seed)
    E, H, I = cfg.E, cfg.H, cfg.I
    codes_gu = rng.integers(0, 256, size=(E, 2 * I, H), dtype=np.uint8)
    codes_dn = rng.integers(0, 256, size=(E, H, I), dtype=np.uint8)
    lut_gu, lut_dn = {}, {}
    for b in BITWIDTHS:
        lut_gu[b] = _draw_luts(rng, E, 2 * I, b)
        lut_dn[b] = _draw_luts(rng, E, H, b)
    q = _draw_q(rng, cfg)
    return Layer(cfg, codes_gu, codes_dn, lut_gu, lut_dn, q, rng.bit_generator.state)


def make_tokens(layer: Layer, T: int) -> Tokens:
    """Hidden states and router logits for T tokens (same weights for every T)."""
    cfg = layer.cfg
    rng = np.random.default_rng()
    rng.bit_generator.state = layer.rng_state
    hidden = float32_to_bf16_bits(rng.standard_normal((T, cfg.H), dtype=np.float32))
    logits = rng.standard_normal((T, cfg.E), dtype=np.float32)
    if cfg.logit_mode == "bias2":
        logits[:, list(cfg.hot)] += np.float32(2.0)
    elif cfg.logit_mode == "zipf":
        logits += np.log(expert_popularity(cfg)).astype(np.float32)[None, :]
    elif cfg.logit_mode != "normal":
        raise ValueError(cfg.logit_mode)
    return Tokens(hidden, logits)


def make_recommit(layer: Layer, seed: int = 1) -> Tuple[np.ndarray, np.ndarray]:
    """A planner's bitwidth recommit: lower a fraction of blocks one rung.

    Picks round(recommit_frac * 2E) blocks uniformly among those whose q is
    above its floor and lowers each to the next bitwidth down the ladder
    3 < 4 < 5 < 6 < 8.  Returns (block_ids int32 [n], new_q int32 [n]) with
    block id 2e+m, ids ascending.
    """
    cfg = layer.cfg
    rng = np.random.default_rng(seed)
    floor = q_floor(cfg).ravel()
    q = layer.q.ravel()
    eligible = np.flatnonzero(q > floor)
    n = int(round(cfg.recommit_frac * q.size))
    n = min(n, eligible.size)
    chosen = np.sort(rng.choice(eligible, size=n, replace=False)).astype(np.int32)
    ladder = list(BITWIDTHS)
    new_q = np.array([ladder[ladder.index(int(q[b])) - 1] for b in chosen], dtype=np.int32)
    return chosen, new_q


def make_sensitivity(layer: Layer, seed: int = 2) -> np.ndarray:
    """Synthetic offline sensitivity per block [2E] (block 2e gate_up, 2e+1
    down): log-normal(0, 1) damage scores standing in for the Hessian-weighted
    scores the planner reads (no trained weights are used)."""
    rng = np.random.default_rng(seed)
    return rng.lognormal(0.0, 1.0, 2 * layer.cfg.E).astype(np.float32)
