"""Parity report: the measured error of the fused layer against the fp64
oracle on every workload and path (the GPU tests assert the bound; this
prints the margin).

Run on a GPU machine from the repository root:
  python tests/parity_report.py

For each (workload, T, path) it prints the relative L2 error of the whole
output (the metric the tests hold to 2e-3) and the largest per-token relative
error.  The oracle runs in a spawn process pool for the large layers.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

from helpers import REL_TOL, host_layer, oracle_out_pool, oracle_route, rel_l2  # noqa: E402
from workloads import gen  # noqa: E402

CASES = [
    ("tiny", 16, ("decode", "prefill")),
    ("qwen15_decode", 1, ("decode",)),
    ("qwen15_decode", 4, ("decode", "prefill")),
    ("qwen15_decode", 8, ("decode",)),
    ("mixtral_decode", 4, ("decode",)),
    ("qwen3_decode", 64, ("decode", "prefill")),
    ("mixtral_prefill", 4096, ("prefill",)),
]


def main():
    import torch
    import any_precision_bitplane_gb300 as pw
    from any_precision_bitplane_gb300.layer import DeviceLayer
    paths = {"decode": pw.PATH_DECODE, "prefill": pw.PATH_PREFILL}
    print("| workload | T | path | rel L2 (whole output) | max per-token rel L2 | bound |")
    print("|---|---|---|---|---|---|")
    for name, T, which in CASES:
        layer = host_layer(name)
        tok = gen.make_tokens(layer, T)
        ids, w = oracle_route(tok, layer.cfg.k)
        dl = DeviceLayer(layer)
        outs = {}
        try:
            hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
            ids_d = torch.from_numpy(ids).cuda()
            w_d = torch.from_numpy(w).cuda()
            for p in which:
                out = pw.moe_forward(hidden, ids_d, w_d, dl.table, dl.I, dl.E, path=paths[p])
                outs[p] = out.cpu().numpy().astype(np.float64)
                if dl.table.status() != pw.PW_OK:
                    raise RuntimeError("device status %d" % dl.table.status())
        finally:
            dl.close()
        ref = oracle_out_pool(name, tok.hidden_bf16, ids, w, layer.q, workers=8)
        ref_norm = np.linalg.norm(ref, axis=1)
        for p in which:
            got = outs[p]
            per_token = np.linalg.norm(got - ref, axis=1) / np.where(ref_norm > 0, ref_norm, 1.0)
            print("| %s | %d | %s | %.2e | %.2e | %.0e |" % (name, T, p, rel_l2(got, ref),
                                                             per_token.max(), REL_TOL))
            sys.stdout.flush()


if __name__ == "__main__":
    main()
