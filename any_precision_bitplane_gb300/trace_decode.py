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
  per CTA      tiles, exit relative to the earliest traced tile start, and
               the idle time from the CTA's exit to the last traced exit (the
               launch's tail).

Run from the repository root:
  python -m any_precision_bitplane_gb300.trace_decode --workload qwen15_decode --T 4
"""
import argparse
import os
import sys

import numpy as np

FIELDS = ("descriptor", "set-up", "columns", "reduction")
CTA_STRIDE = 19   # traced CTAs: block index = CTA_STRIDE * trace slot


def summarize(tile, cta):
    """Medians of the record that pw_debug_decode_trace returns (tile uint64
    [16, 32, 10], cta uint64 [16, 2]).  Returns a dict: `per_q` maps each
    bitwidth to its traced tiles, the medians of the four phases (cycles),
    of the set-up's three parts, of the pair count and of the tile duration
    (us); `all` holds the same over every traced tile plus `shares` (each
    phase's median over the sum of the four medians); `ctas` lists (CTA, SM,
    tiles, exit us, idle us) per traced CTA, idle being the time from its exit
    to the last traced exit; `span_us` runs from the first traced tile start
    to that exit."""
    tile = np.asarray(tile, dtype=np.int64)
    cta = np.asarray(cta, dtype=np.int64)
    done = (tile[:, :, 0] > 0) & (tile[:, :, 1] > 0)
    q = tile[:, :, 6] & 255
    pairs = tile[:, :, 6] >> 8
    dur_us = (tile[:, :, 1] - tile[:, :, 0]) / 1e3

    def stats(m):
        med = [float(np.median(tile[:, :, 2 + f][m])) for f in range(4)]
        return {"tiles": int(m.sum()), "phases": med,
                "setup_parts": [float(np.median(tile[:, :, f][m])) for f in (7, 8, 9)],
                "pairs": float(np.median(pairs[m])), "tile_us": float(np.median(dur_us[m]))}

    out = {"per_q": {int(qq): stats(done & (q == qq)) for qq in sorted(set(q[done].tolist()))}}
    out["all"] = stats(done)
    tot = sum(out["all"]["phases"])
    out["all"]["shares"] = [p / tot for p in out["all"]["phases"]]
    t0 = tile[:, :, 0][tile[:, :, 0] > 0].min()
    traced = np.nonzero(cta[:, 0] > 0)[0]
    end = cta[traced, 1].max()
    out["ctas"] = [(CTA_STRIDE * int(c), int(cta[c, 0]) - 1, int(done[c].sum()),
                    (cta[c, 1] - t0) / 1e3, (end - cta[c, 1]) / 1e3) for c in traced]
    out["span_us"] = (end - t0) / 1e3
    return out


def print_summary(sm):
    print("%3s %6s %11s %9s %9s %10s %8s %10s" % ("q", "tiles", "descriptor", "set-up",
                                                   "columns", "reduction", "pairs",
                                                   "tile_us"))
    rows = [("%3d" % qq, st) for qq, st in sm["per_q"].items()] + [("all", sm["all"])]
    for label, st in rows:
        ph = st["phases"]
        print("%3s %6d %11.0f %9.0f %9.0f %10.0f %8.1f %10.2f" % (
            label, st["tiles"], ph[0], ph[1], ph[2], ph[3], st["pairs"], st["tile_us"]))
    print("shares of a median tile's thread-0 cycles: " + ", ".join(
        "%s %.0f%%" % (FIELDS[f], 100.0 * sm["all"]["shares"][f]) for f in range(4)))
    print("set-up parts per q (median cycles per tile, summed over its passes): "
          "issue, LUT wait + table build, barrier")
    for qq, st in sm["per_q"].items():
        print("  q=%d: %s" % (qq, ", ".join("%.0f" % v for v in st["setup_parts"])))
    print("%4s %4s %6s %9s %9s" % ("CTA", "SM", "tiles", "exit_us", "idle_us"))
    for c, smid, n, ex, idle in sm["ctas"]:
        print("%4d %4d %6d %9.2f %9.2f" % (c, smid, n, ex, idle))
    idle = [c[4] for c in sm["ctas"]]
    if idle:
        print("traced span %.2f us; CTAs idle before the last exit: median %.2f us, max %.2f us"
              % (sm["span_us"], float(np.median(idle)), float(np.max(idle))))


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
    dl.close()
    if not (tile[:, :, 0] > 0).any():
        raise SystemExit("no traced tile (is the call on the decode path?)")
    print("workload %s, T=%d: decode gate_up tiles of CTAs 0, 19, ..., 285 "
          "(SM cycles of thread 0; durations in us)" % (args.workload, args.T))
    print_summary(summarize(tile, cta))


if __name__ == "__main__":
    main()
