"""Pipeline trace of the tensor-core gate_up GEMM (a measurement tool).

Needs the traced library: `python any_precision_bitplane_gb300/build.py --trace`
writes libpw_trace.so (the same sources with -DPW_TRACE).  This tool loads that
library instead of libpw.so, runs a few forward calls of a workload, and
summarises the %globaltimer stamps that the last gate_up GEMM launch left for
its CTAs 0, 10, ..., 150 (pw_debug_gemm_trace), with the SM each one ran on:

  per k-step   the MMA issuer's interval between issued stages; the slack
               between a dequant set announcing a stage and the issuer finding
               it full (positive: the stage waited for the issuer);
  per tile     MMA phase (accumulator free -> last commit), epilogue (drain),
               the gap the issuer spends waiting for the next accumulator, and
               the dequant warps' LUT load.

Run from the repository root:
  python -m any_precision_bitplane_gb300.trace_gemm --workload mixtral_prefill --T 2048
  python -m any_precision_bitplane_gb300.trace_gemm --workload qwen3_decode --T 64
"""
import argparse
import os
import sys

import numpy as np


INTERVALS = ("kstep", "slack", "mma", "epi", "idle", "lut")


def cta_intervals(s, t):
    """One traced CTA's intervals (ns) from its k-step stamps s [steps, 4]
    (issuer found full, issued, announced, producer found empty) and tile
    stamps t [tiles, 6] (MMA start, last commit, epilogue start and end, LUT
    load start and end); 0 marks a stamp not reached.  kstep: the issue
    interval between consecutive issued k-steps, without the gaps that span a
    tile boundary (more than 4 x the median: they hold the epilogue); slack:
    how long an announced stage waited for the issuer; mma, epi, lut: per
    tile; idle: from a tile's last commit to the next tile's MMA start."""
    done = np.nonzero((s[:, 0] > 0) & (s[:, 1] > 0))[0]
    rows = np.nonzero(t[:, 0] > 0)[0]
    issued = set(done.tolist())
    gaps = [int(s[i + 1, 1] - s[i, 1]) for i in done[:-1] if (i + 1) in issued]
    out = {
        "tiles": int(rows.size),
        "slack": [int(s[i, 0] - s[i, 2]) for i in done if s[i, 2] > 0],
        "mma": [int(t[j, 1] - t[j, 0]) for j in rows if t[j, 1] > 0],
        "epi": [int(t[j, 3] - t[j, 2]) for j in rows if t[j, 2] > 0 and t[j, 3] > 0],
        "idle": [int(t[j + 1, 0] - t[j, 1]) for j in rows
                 if j + 1 < t.shape[0] and t[j + 1, 0] > 0 and t[j, 1] > 0],
        "lut": [int(t[j, 5] - t[j, 4]) for j in rows if t[j, 4] > 0 and t[j, 5] > 0],
    }
    if out["mma"] and gaps:
        cut = np.median(gaps) * 4
        gaps = [g for g in gaps if g < cut]
    out["kstep"] = gaps
    return out


def summarize(step, tile, smid, cta_stride=10):
    """Per traced CTA (smid > 0): (CTA, SM, its intervals); and the medians of
    each interval over all traced CTAs (None where none was recorded)."""
    step = np.asarray(step, dtype=np.int64)
    tile = np.asarray(tile, dtype=np.int64)
    per_cta, agg = [], {k: [] for k in INTERVALS}
    for c in range(step.shape[0]):
        if smid[c] == 0:
            continue
        iv = cta_intervals(step[c], tile[c])
        per_cta.append((cta_stride * c, int(smid[c]) - 1, iv))
        for k in INTERVALS:
            agg[k] += iv[k]
    medians = {k: (float(np.median(v)) if v else None) for k, v in agg.items()}
    return per_cta, medians


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="mixtral_prefill")
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--dump", type=int, default=-1,
                    help="also print the raw k-step stamps of this trace slot (CTA = 10 x slot)")
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
    for _ in range(args.calls):
        pw.moe_forward(hidden, ids, w, dl.table, cfg.I, cfg.E, out=out, workspace=ws)
    torch.cuda.synchronize()
    step, tile, smid, dq = pw.debug_gemm_trace()
    dq = dq.astype(np.int64)
    step = step.astype(np.int64)
    tile = tile.astype(np.int64)
    print("workload %s, T=%d: gate_up GEMM stamps of CTAs 0, 10, ..., 150 (ns unless noted)"
          % (args.workload, args.T))
    per_cta, medians = summarize(step, tile, smid)
    print("%4s %4s %6s %9s %9s %9s %9s %9s %9s %9s" %
          ("CTA", "SM", "tiles", "kstep_md", "kstep_p90", "slack_md", "mma_us", "epi_us",
           "idle_us", "lut_us"))

    def md(v, scale=1.0):
        return "%9.1f" % (np.median(v) / scale) if len(v) else "%9s" % "-"
    for cta, sm, iv in per_cta:
        gaps = iv["kstep"]
        print("%4d %4d %6d %s %s %s %s %s %s %s" % (
            cta, sm, iv["tiles"], md(gaps),
            ("%9.1f" % np.percentile(gaps, 90)) if gaps else "%9s" % "-", md(iv["slack"]),
            md(iv["mma"], 1e3), md(iv["epi"], 1e3), md(iv["idle"], 1e3), md(iv["lut"], 1e3)))
    if 0 <= args.dump < step.shape[0] and smid[args.dump]:
        s = step[args.dump]
        t0 = s[0, 0]
        print("raw k-step stamps of CTA %d, ns from its first: issuer found full, issued, "
              "dequant set announced (its first warp), token producer found the stage free; "
              "then over the set's 8 warps (first / last): plane words arrived, transpose done, "
              "release seen, announced"
              % (args.dump * 10))
        d = dq[args.dump]
        for i in range(min(48, s.shape[0])):
            cols = [[v for v in d[i, :, k] if v] for k in (2, 3, 0, 1)]
            extra = " ".join("%8d %8d" % (min(c) - t0, max(c) - t0) for c in cols) \
                if all(cols) else ""
            print("%4d %s  %s" % (i, " ".join("%8d" % (v - t0) if v else "       -" for v in s[i]),
                                  extra))
    print("all traced CTAs: k-step interval median %.0f ns; stage ready %.0f ns before the "
          "issuer reached it (median); tile MMA phase %.1f us, epilogue %.1f us, issuer idle "
          "between tiles %.1f us, LUT load %.1f us (medians)" % (
              medians["kstep"], medians["slack"], medians["mma"] / 1e3, medians["epi"] / 1e3,
              medians["idle"] / 1e3, medians["lut"] / 1e3))


if __name__ == "__main__":
    main()
