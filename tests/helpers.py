"""Shared helpers for the GPU parity tests: seeded layers, the oracle's
expected outputs (in a spawn process pool for the large layers) and the
rel-L2 tolerance the layer output is held to."""
import functools
import multiprocessing as mp
import os

import numpy as np

from oracle import apl, moe
from workloads import configs, gen

# Relative L2 error bound for the fp32 layer output (norm of the error over
# norm of the oracle's fp64 output, per tensor).
REL_TOL = 2e-3


@functools.lru_cache(maxsize=4)
def host_layer(name, seed=0):
    return gen.make_layer(configs.config_by_name(name), seed)


def oracle_blocks(layer, q=None):
    """block(e, m) for the oracle: planes packed by the oracle from the codes,
    LUT and bitwidth as committed (q [E, 2] overrides layer.q)."""
    qs = layer.q if q is None else np.asarray(q)
    cache = {}

    def block(e, m):
        key = (e, m)
        if key not in cache:
            codes, luts, _ = layer.block(e, m)
            qq = int(qs[e, m])
            cache[key] = (apl.pack_bitplanes(codes), luts[qq], qq)
        return cache[key]
    return block


def oracle_route(tokens, k):
    ids, w = moe.route_topk(tokens.logits, k)
    return ids, w.astype(np.float32)


def oracle_out(layer, hidden, ids, w, q=None, tokens=None, drop_experts=()):
    """Expected layer output (fp64).  Pairs routed to drop_experts contribute 0."""
    block = oracle_blocks(layer, q)
    experts = [e for e in range(layer.cfg.E) if e not in set(drop_experts)]
    y = moe.expert_outputs(hidden, ids, block, layer.cfg.E, experts=experts, tokens=tokens)
    return _combine_with_drops(y, ids, w, layer.cfg.H, tokens)


def _combine_with_drops(y, ids, w, H, tokens):
    T, k = ids.shape
    for t in (range(T) if tokens is None else tokens):
        for j in range(k):
            y.setdefault(int(t) * k + j, np.zeros(H))
    return moe.combine(y, w, H, tokens=tokens)


def _pool_worker(args):
    name, seed, hidden, ids, q, experts, tokens = args
    layer = gen.make_layer(configs.config_by_name(name), seed)
    block = oracle_blocks(layer, q)
    return moe.expert_outputs(hidden, ids, block, layer.cfg.E, experts=experts, tokens=tokens)


def oracle_out_pool(name, hidden, ids, w, q, seed=0, tokens=None, workers=4):
    """oracle_out for a named config, experts spread over a spawn pool; each
    worker regenerates the layer from its seed."""
    cfg = configs.config_by_name(name)
    routed = sorted(set(int(e) for e in np.unique(ids)))
    chunks = [routed[i::workers] for i in range(workers) if routed[i::workers]]
    ctx = mp.get_context("spawn")
    # share the host cores between the workers' BLAS instead of oversubscribing
    threads = str(max(1, (os.cpu_count() or 1) // len(chunks)))
    saved = {v: os.environ.get(v) for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    for v in saved:
        os.environ[v] = threads
    try:
        with ctx.Pool(len(chunks)) as pool:
            parts = pool.map(_pool_worker, [(name, seed, hidden, ids, q, c, tokens) for c in chunks])
    finally:
        for v, old_v in saved.items():
            if old_v is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old_v
    y = {}
    for part in parts:
        y.update(part)
    return _combine_with_drops(y, ids, w, cfg.H, tokens)


def rel_l2(got, ref):
    return moe.rel_l2(got, ref)
