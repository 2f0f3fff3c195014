"""Greedy damage-per-byte bitwidth planner (oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: PagedWeight, "Core components" 2 (quality-aware runtime planner):
each possible bitwidth cut gets a damage score; when a memory target is set,
the planner greedily takes the cuts with the least damage per byte saved;
frequently routed ("hot") experts are protected by a higher bitwidth floor and
a damage multiplier.

Readings (the pages give no formulas):
  * a cut lowers one block by one rung of the ladder 8 > 6 > 5 > 4 > 3;
  * the relative error of a b-bit quantiser is 4^-b, so lowering b to b'
    costs damage = sensitivity * m_e * (4^-b' - 4^-b) and saves
    (b - b') * bytes_per_bit bytes (the freed tail planes);
  * expert e's share is its routing mass over the total; it is hot when the
    share exceeds 1/E, which sets its floor to hot_floor (others: 3); its
    multiplier is m_e = max(1, E * share);
  * the planner takes, one at a time, the cut with the least damage per byte
    (ties: the lower block id) until the target is met or no cut is left.
Arithmetic is in fp64 on the fp32 inputs; the routing-mass total is summed in
expert order.
"""
from typing import List, Sequence, Tuple

import numpy as np

LADDER = (3, 4, 5, 6, 8)


def quant_error(b: int) -> float:
    return 1.0 / float(4 ** b)


def plan_recommit(q_now: Sequence[int], sensitivity, bytes_per_bit: Sequence[int], routing_mass,
                  hot_floor: int, bytes_to_free: int, trace: List = None
                  ) -> Tuple[List[int], List[int], int]:
    """Returns (block ids whose bitwidth changed, ascending; their new
    bitwidths; bytes saved).  `trace`, if given, receives (ratio, block, to)
    for every cut in the order taken."""
    n = len(q_now)
    E = n // 2
    sens = [float(np.float32(s)) for s in sensitivity]
    mass = [float(np.float32(m)) for m in routing_mass]
    total = 0.0
    for m in mass:
        total += m
    floors, mults = [], []
    for i in range(n):
        m = mass[i // 2]
        hot = total > 0.0 and m * E > total
        floors.append(hot_floor if hot else LADDER[0])
        scaled = m * E / total if total > 0.0 else 1.0
        mults.append(scaled if scaled > 1.0 else 1.0)
    q = list(int(x) for x in q_now)

    def next_cut(i):
        r = LADDER.index(q[i])
        if r == 0:
            return None
        to = LADDER[r - 1]
        if to < floors[i]:
            return None
        nbytes = (q[i] - to) * int(bytes_per_bit[i])
        if nbytes <= 0:
            return None
        damage = sens[i] * mults[i] * (quant_error(to) - quant_error(q[i]))
        return damage / float(nbytes), to, nbytes

    freed = 0
    while freed < bytes_to_free:
        best, best_i = None, -1
        for i in range(n):
            c = next_cut(i)
            if c is not None and (best is None or c[0] < best[0]):
                best, best_i = c, i
        if best is None:
            break
        q[best_i] = best[1]
        freed += best[2]
        if trace is not None:
            trace.append((best[0], best_i, best[1]))
    ids = [i for i in range(n) if q[i] != int(q_now[i])]
    return ids, [q[i] for i in ids], freed
