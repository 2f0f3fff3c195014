"""Per-tile phase trace of the decode gate_up kernel (a measurement tool).

Needs the traced library: `python any_precision_bitplane_gb300/build.py --trace`
writes libpw_trace.so (the same sources with -DPW_TRACE).  This tool loads that
library instead of libpw.so, runs a few decode calls of a workload (L2 flushed
before each, so the weights come from HBM), and summarises what the last
gate_up launch recorded for its CTAs 0, 19, ..., 285 (pw_debug_decode_trace):

  per q        tiles traced, median SM cycles of thread 0 on the slot
               descriptor, the passes' set-up (LUT fetch, first ring copies,
               table build), the column loops and the reduction + h stores,
               and the median tile duration;
  per CTA      tiles, first tile start and exit relative to the earliest
               traced start, and the idle time from the CTA's exit to the last
               traced exit (the launch's tail).

Run from the repository root:
  python -m any_precision_bitplane_gb300.trace_decode --workload qwen15_decode --T 4
"""
import argparse
import os
import sys

import numpy as np

FIELDS = ("descriptor", "set-up", "columns", "reduction")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen15_decode")
    ap.add_argument("--T", type=int, default=4)
    ap.add_argument("--calls", type=int, default=5)
    args = ap.parse_args()

    sys.path.insert(0, os.getcwd())
    import torch
    import any_precision_bitplane_gb300 as pw
    from any_precision_bitplane_gb300.layer import DeviceLayer
    from workloads import configs, gen

    if not os.path.exists(pw.TRACE_LIB_PATH):
        raise SystemExit("build the traced library first: "
                         "python any_precision_bitplane_gb300/build.py --trace")
    pw.LIB_PATH = pw.TRACE_LIB_PATH
    pw.lib()

    cfg = configs.config_by_name(args.workload)
    layer = gen.make_layer(cfg, 0)
    dl = DeviceLayer(layer)
    tok = gen.make_tokens(layer, args.T)
    ids, w = pw.route_topk(torch.from_numpy(tok.logits).cuda(), cfg.k)
    hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).cuda()
    out = torch.empty((args.T, cfg.H), dtype=torch.float32, device="cuda")
    ws = torch.empty(pw.workspace_bytes(args.T, cfg.H, cfg.I, cfg.E, cfg.k), dtype=torch.uint8,
                     device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")   # > 4 x L2
    for _ in range(args.calls):
        flush.fill_(1)
        pw.moe_forward(hidden, ids, w, dl.table, cfg.I, cfg.E, out=out, workspace=ws,
                       path=pw.PATH_DECODE)
    torch.cuda.synchronize()
    tile, cta = pw.debug_decode_trace()
    tile = tile.astype(np.int64)
    cta = cta.astype(np.int64)

    starts = tile[:, :, 0][tile[:, :, 0] > 0]
    if starts.size == 0:
        raise SystemExit("no traced tile (is the call on the decode path?)")
    t0 = starts.min()
    print("workload %s, T=%d: decode gate_up tiles of CTAs 0, 19, ..., 285 "
          "(SM cycles of thread 0; durations in us)" % (args.workload, args.T))
    print("%3s %6s %11s %9s %9s %10s %8s %10s" % ("q", "tiles", "descriptor", "set-up",
                                                   "columns", "reduction", "pairs",
                                                   "tile_us"))
    done = (tile[:, :, 1] > 0) & (tile[:, :, 0] > 0)
    q = tile[:, :, 6] & 255
    pairs = tile[:, :, 6] >> 8
    allq = []
    for qq in sorted(set(q[done].tolist())):
        m = done & (q == qq)
        med = [np.median(tile[:, :, 2 + f][m]) for f in range(4)]
        dur = np.median((tile[:, :, 1] - tile[:, :, 0])[m]) / 1e3
        print("%3d %6d %11.0f %9.0f %9.0f %10.0f %8.1f %10.2f" % (
            qq, m.sum(), med[0], med[1], med[2], med[3], np.median(pairs[m]), dur))
        allq.append(m)
    m = done
    med = [np.median(tile[:, :, 2 + f][m]) for f in range(4)]
    tot = sum(med)
    print("all %6d %11.0f %9.0f %9.0f %10.0f %8.1f %10.2f" % (
        m.sum(), med[0], med[1], med[2], med[3], np.median(pairs[m]),
        np.median((tile[:, :, 1] - tile[:, :, 0])[m]) / 1e3))
    print("shares of a median tile's thread-0 cycles: " + ", ".join(
        "%s %.0f%%" % (FIELDS[f], 100.0 * med[f] / tot) for f in range(4)))
    print("set-up parts per q (median cycles per tile, summed over its passes): "
          "issue, LUT wait + table build, barrier")
    for qq in sorted(set(q[done].tolist())):
        mq = done & (q == qq)
        print("  q=%d: %s" % (qq, ", ".join("%.0f" % np.median(tile[:, :, f][mq])
                                            for f in (7, 8, 9))))

    exits = cta[:, 1][cta[:, 0] > 0]
    end = exits.max() if exits.size else 0
    print("%4s %4s %6s %10s %9s %9s" % ("CTA", "SM", "tiles", "start_us", "exit_us", "idle_us"))
    idle = []
    for c in range(cta.shape[0]):
        if cta[c, 0] == 0:
            continue
        n = int(done[c].sum())
        st = tile[c, 0, 0] - t0 if tile[c, 0, 0] > 0 else 0
        ex = cta[c, 1] - t0
        idle.append((end - cta[c, 1]) / 1e3)
        print("%4d %4d %6d %10.2f %9.2f %9.2f" % (19 * c, cta[c, 0] - 1, n, st / 1e3, ex / 1e3,
                                                    (end - cta[c, 1]) / 1e3))
    if idle:
        print("traced span %.2f us; CTAs idle before the last exit: median %.2f us, max %.2f us"
              % ((end - t0) / 1e3, float(np.median(idle)), float(np.max(idle))))
    dl.close()


if __name__ == "__main__":
    main()
