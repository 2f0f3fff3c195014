"""CPU oracle for the fused mixed-precision MoE layer over Any-Precision bitplanes.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: it is used by tests/, by the smoke check in __graft_entry__.py and by
the CPU-baseline leg of bench.py.  It shares no code with the CUDA library.

It is a plain, slow, obviously-correct restatement, in NumPy with fp64 for
every floating-point step, of what the layer computes:

* apl.py  -- the overlay bitplane format with per-row lookup tables
             (PagedWeight, "Core components" 1, Paged Weight representation:
             weights kept as stacked bitplanes plus LUTs, a b-bit model read
             from the top b planes).
* moe.py  -- top-k routing, the token-to-expert permutation, the expert MLP
             (gate_up, SiLU(gate) * up, down) and the weighted top-k combine
             (PagedWeight, "Core components" 3, fused mixed-precision kernel:
             every linear block read at its own committed bitwidth q_i).

Readings taken where the pages are silent (bit order, plane order, layout,
gate/up row split, tie-breaking) are stated in each function's docstring.

Pinning status (what each function is checked against in tests/):
  pack_bitplanes / unpack_top  -- worked examples in tests/golden/, the
                                  identity idx_b == code >> (8-b), round trip.
  dequant                      -- b=8 reproduces the LUT weights; integer and
                                  row-tagged LUT closed forms.
  route_topk                   -- weights renormalise to 1; ids equal a
                                  brute-force selection; k=1/k=2 closed forms.
  permute                      -- pure-Python bucket loop; inverse identity.
  moe_forward                  -- explicit triple-loop brute force on tiny
                                  inputs (computed from the codes, not the
                                  planes); one-hot and constant-LUT closed forms.
  rel_l2                       -- closed-form values worked by hand from the
                                  metric's definition (tests/golden/).
"""
from . import apl, moe  # noqa: F401
