#!/usr/bin/env python
"""Throughput of the fused mixed-precision MoE layer (PagedWeight) on GB300.

One step = one pw_moe_forward call over one batch of the workload: every
routed expert's gate_up and down blocks read at their committed bitwidths
from the overlay bitplanes + per-row LUTs, SiLU gating, and the weighted
top-k combine.  Inputs are synthetic and seeded (workloads/), resident in
HBM before the timed region; L2 is defeated by rotating independent copies
of the layer (planes, LUTs and page table each), so every step reads its
weights from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--T T]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica of the layer (the layer has no cross-GPU exchange); value sums the
tokens of all ranks over the slowest rank's time.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

# The CPU baseline's BLAS (NumPy's fp64 matmuls inside the oracle) runs on
# every host core; the thread count is fixed here, before NumPy loads, so
# that the reported core count is the one actually used.
HOST_CORES = os.cpu_count() or 1
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_var, str(HOST_CORES))

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
DECODE_LAUNCHES_PER_CALL = 3   # prep (grouping, activation forms), gate_up + SiLU, down + combine
HYBRID_MIN_TOKENS = 16         # calls of this many tokens also launch the heavy experts'
                               # gather and two GEMM kernels (when the shape suits them)


def launches_per_call(cfg, T):
    """Kernel launches of one decode call of the library (its own kernels only)."""
    hybrid = (T >= HYBRID_MIN_TOKENS and cfg.H % 128 == 0 and cfg.I % 64 == 0 and cfg.E <= 1024)
    return DECODE_LAUNCHES_PER_CALL + (3 if hybrid else 0)
HBM_FALLBACK_GBS = 6800.0
KERNEL_SOURCES = ("any_precision_bitplane_gb300/csrc/pw_decode.cu",
                  "any_precision_bitplane_gb300/csrc/pw_prefill.cu")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", default="qwen15_decode")
    ap.add_argument("--T", type=int, default=4, help="tokens per step (decode batch)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the other batch sizes")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--copies", type=int, default=0,
                    help="layer copies to rotate (0: enough to exceed 2x L2)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill section and print its JSON")
    ap.add_argument("--prefill-tokens", type=int, default=0,
                    help="tokens of the prefill section (0: the workload's 4096)")
    ap.add_argument("--uniform-q", type=int, default=0, choices=(0, 3, 4, 5, 6, 8),
                    help="commit every block of the timed workload at this bitwidth "
                         "(0: the workload's own mix); for per-bitwidth measurements")
    return ap.parse_args()


SHAPE_NAMES = {"qwen15_decode": "Qwen1.5-MoE-A2.7B-shaped layer",
               "mixtral_decode": "Mixtral-8x7B-shaped layer",
               "qwen3_decode": "Qwen3-30B-A3B-shaped layer",
               "tiny": "tiny layer"}


def metric_name(workload):
    return "MoE-layer tokens/s (decode, %s)" % SHAPE_NAMES.get(workload, workload)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def slowest_rank_seconds(seconds, world, device=None):
    """The job's time for a quantity each rank measured on its own: the
    maximum over ranks (an all-reduce with MAX over the default process group
    when world > 1; `device` is where the reduced tensor lives, the rank's GPU
    under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(seconds)
    import torch
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, seconds, world, device=None):
    """Whole-job throughput: the tokens of all ranks over the slowest rank's
    time (weak scaling: each rank processes its own tokens_per_rank)."""
    return tokens_per_rank * world / slowest_rank_seconds(seconds, world, device)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def tensor_peak():
    """Dense fp16 tensor peak for a kernel timed alone: the measured bf16 burst
    figure (fp16 and bf16 have the same nominal dense rate), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst, fp16 = bf16 nominal)"
    except Exception:
        return 1900.0, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload, T):
    """DRAM bytes (read + write) per launch of `kernel` on this workload from
    the committed ncu summary, if it was taken on the current kernel sources;
    else None.  Line format: kernel workload T=<T> <bytes> <source sha>."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if (len(parts) == 5 and parts[0] == kernel and parts[1] == workload
                        and parts[2] == "T=%d" % T and parts[4] == kernel_source_sha()):
                    return float(parts[3])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 100 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for ts, r in self.rows if t0 - 0.15 <= ts <= t1 + 0.15] or [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = set()
        sm, mx = [], []
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- native arm

def setup_workload(name, T, device, copies=0, uniform_q=0):
    import dataclasses
    import torch
    import any_precision_bitplane_gb300 as pw
    from any_precision_bitplane_gb300.layer import DeviceLayer
    from workloads import configs, gen

    cfg = configs.config_by_name(name)
    layer = gen.make_layer(cfg, 0)
    if uniform_q:   # every block committed at one bitwidth (a per-bitwidth measurement)
        layer = dataclasses.replace(layer, q=np.full_like(layer.q, uniform_q))
    base = DeviceLayer(layer, device=device)
    tok = gen.make_tokens(layer, T)
    logits = torch.from_numpy(tok.logits).to(device)
    ids, wts = pw.route_topk(logits, cfg.k)          # the library's router, on the device
    hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).to(device)
    torch.cuda.synchronize(device)
    ids_host = ids.cpu().numpy()
    weight_bytes = base.routed_bytes(ids_host)
    step_bytes = weight_bytes + T * cfg.H * 2 + T * cfg.k * 8 + T * cfg.H * 4
    if copies <= 0:
        copies = max(2, math.ceil(2 * L2_BYTES / max(weight_bytes, 1)))
    layers = [base] + [base.clone() for _ in range(copies - 1)]
    host = {"hidden": tok.hidden_bf16.view(np.int16), "ids": ids_host,
            "wts": wts.cpu().numpy()}
    return cfg, layer, layers, hidden, ids, wts, step_bytes, weight_bytes, host


def time_device(pw, cfg, layers, hidden, ids, wts, steps, warmup, stream):
    import torch
    T = hidden.shape[0]
    out = torch.empty((T, cfg.H), dtype=torch.float32, device=hidden.device)
    ws = torch.empty(max(pw.workspace_bytes(T, cfg.H, cfg.I, cfg.E, cfg.k), 256),
                     dtype=torch.uint8, device=hidden.device)
    L = len(layers)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            pw.moe_forward(hidden, ids, wts, layers[i % L].table, cfg.I, cfg.E, out=out,
                           workspace=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                pw.moe_forward(hidden, ids, wts, layers[i % L].table, cfg.I, cfg.E, out=out,
                               workspace=ws)
        g.replay()                     # instantiation/upload, untimed
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        return g, start, stop, out


def time_dominant(pw, cfg, layers, hidden, ids, wts, steps, stream):
    """Average duration of the call's dominant kernel: the library records a
    pair of CUDA events around it (on the launching stream) in every step of
    a captured graph of `steps` calls; returns milliseconds per launch."""
    import torch
    T = hidden.shape[0]
    out = torch.empty((T, cfg.H), dtype=torch.float32, device=hidden.device)
    ws = torch.empty(max(pw.workspace_bytes(T, cfg.H, cfg.I, cfg.E, cfg.k), 256),
                     dtype=torch.uint8, device=hidden.device)
    L = len(layers)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for b, a in evs:        # create the events before capture
            b.record(stream)
            a.record(stream)
        pw.moe_forward(hidden, ids, wts, layers[0].table, cfg.I, cfg.E, out=out, workspace=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g, stream=stream):
                for i in range(steps):
                    pw.set_timing_events(*evs[i])
                    pw.moe_forward(hidden, ids, wts, layers[i % L].table, cfg.I, cfg.E, out=out,
                                   workspace=ws)
        finally:
            pw.set_timing_events(None, None)
        g.replay()
        torch.cuda.synchronize()
    total = sum(b.elapsed_time(a) for b, a in evs)
    del g
    return total / steps


def time_e2e(pw, cfg, layers, host, steps, warmup, device):
    """End to end through the C ABI with HOST buffers: every step hands
    pw_moe_forward pinned host pointers for hidden, topk ids, topk weights and
    out, so the step's inputs travel host -> device and its result device ->
    host inside the call (the kernels read and write the pinned pages directly
    over the CPU-GPU link; the pointers are valid on the device under unified
    addressing).  The K steps are captured in one CUDA graph and timed on the
    wall clock around its replay; the last output is checked against the same
    call on device buffers."""
    import ctypes
    import torch
    T = host["hidden"].shape[0]
    k = host["ids"].shape[1]
    h_hidden = torch.from_numpy(host["hidden"].copy()).pin_memory()
    h_ids = torch.from_numpy(host["ids"].astype(np.int32)).pin_memory()
    h_wts = torch.from_numpy(host["wts"].astype(np.float32)).pin_memory()
    h_out = torch.zeros((T, cfg.H), dtype=torch.float32).pin_memory()
    ws_bytes = max(pw.workspace_bytes(T, cfg.H, cfg.I, cfg.E, cfg.k), 256)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    shape = pw.MoeShape(T, cfg.H, cfg.I, cfg.E, k)
    L = len(layers)
    stream = torch.cuda.Stream(device)
    lib = pw.lib()

    def step(i):
        rc = lib.pw_moe_forward(ctypes.byref(shape), ctypes.c_void_p(h_hidden.data_ptr()),
                                ctypes.c_void_p(h_ids.data_ptr()),
                                ctypes.c_void_p(h_wts.data_ptr()), layers[i % L].table.handle,
                                ctypes.c_void_p(h_out.data_ptr()),
                                ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(ws_bytes),
                                ctypes.c_void_p(stream.cuda_stream))
        if rc != pw.PW_OK:
            raise RuntimeError("pw_moe_forward (host buffers): %s" % pw.last_error())

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                step(i)
        g.replay()                     # instantiation/upload, untimed
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        g.replay()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    ref = pw.moe_forward(h_hidden.to(device), h_ids.to(device), h_wts.to(device),
                         layers[(steps - 1) % L].table, cfg.I, cfg.E)
    if not torch.equal(ref.cpu(), h_out):
        raise RuntimeError("e2e: the host-buffer output differs from the device-buffer call")
    del g
    bi = h_hidden.numel() * 2 + h_ids.numel() * 4 + h_wts.numel() * 4
    return dt, bi, h_out.numel() * 4


def _oracle_setup(name, T):
    """The oracle's inputs: routing from its router, every block encoded once
    into bitplanes (storage, done before timing as on the GPU side)."""
    from oracle import apl, moe
    from workloads import configs, gen
    cfg = configs.config_by_name(name)
    layer = gen.make_layer(cfg, 0)
    tok = gen.make_tokens(layer, T)
    ids, w = moe.route_topk(tok.logits, cfg.k)
    encoded = {}
    for e in sorted(set(int(x) for x in np.unique(ids))):
        for m in (0, 1):
            codes, luts, q = layer.block(e, m)
            encoded[(e, m)] = (apl.pack_bitplanes(codes), luts[q], q)
    return cfg, tok, ids, w.astype(np.float32), (lambda e, m: encoded[(e, m)])


def blas_threads():
    """Threads NumPy's BLAS uses: read back through threadpoolctl where it is
    installed, else the thread-count variable set before NumPy loaded."""
    try:
        from threadpoolctl import threadpool_info
        n = [int(i["num_threads"]) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n), "threadpoolctl"
    except Exception:
        pass
    return int(os.environ.get("OPENBLAS_NUM_THREADS", "1")), "OPENBLAS_NUM_THREADS"


def host_cores_entry():
    n, how = blas_threads()
    return {"cores": n, "cpu_count": HOST_CORES, "blas_threads": n, "blas_threads_from": how}


def cpu_baseline(name, T, budget_s=20.0):
    """The oracle as it stands, on host cores, over a bounded sample: whole
    decode batches (stops after ~budget_s or 3 batches)."""
    from oracle import moe
    cfg, tok, ids, w, block = _oracle_setup(name, T)
    done, calls, t0 = 0, 0, time.perf_counter()
    while True:
        moe.moe_forward(tok.hidden_bf16, ids, w, block, cfg.E)
        done += T
        calls += 1
        if time.perf_counter() - t0 > budget_s or calls >= 3:
            break
    dt = time.perf_counter() - t0
    entry = {"value": done / dt, "unit": "tokens/s", "kind": "oracle",
             "sample": "%d full forward(s) of the T=%d batch: fp64 NumPy in one process "
                       "(top-q unpack + LUT dequant of every routed block, matmuls on the "
                       "BLAS threads, combine; blocks encoded before timing)" % (calls, T)}
    entry.update(host_cores_entry())
    return entry


def hidden_bytes(cfg, T):
    """bf16 hidden states of one batch."""
    return T * cfg.H * 2


def decode_config(pw, name, T, device, stream, steps, warmup, recommit=False):
    """Tokens/s and achieved bytes/s of another decode workload (same timing
    method as the headline; a parity-test configuration, reported as context)."""
    import torch
    from workloads import gen
    cfg, layer, layers, hidden, ids, wts, step_bytes, weight_bytes, _ = \
        setup_workload(name, T, device)
    peak, _ = measured_peaks()
    res = {}
    phases = ["before recommit", "after recommit"] if recommit else [""]
    for ph in phases:
        if ph == "after recommit":
            blocks, new_q = gen.make_recommit(layer)
            for x in layers:
                x.commit(blocks, new_q)
            torch.cuda.synchronize()
            step_bytes = (layers[0].routed_bytes(ids.cpu().numpy()) + T * cfg.H * 2 +
                          T * cfg.k * 8 + T * cfg.H * 4)
        g, s0, s1, _ = time_device(pw, cfg, layers, hidden, ids, wts, steps, warmup, stream)
        with torch.cuda.stream(stream):
            s0.record(stream)
            g.replay()
            s1.record(stream)
        torch.cuda.synchronize()
        ms = s0.elapsed_time(s1)
        gbs = step_bytes / (ms / 1e3 / steps) / 1e9
        entry = {"tokens_per_s": T * steps / (ms / 1e3), "us_per_step": ms * 1e3 / steps,
                 "GB_per_s": gbs, "frac": gbs / peak, "bytes_per_step": step_bytes}
        if ph:
            res[ph] = entry
        else:
            res = entry
        del g
    for x in layers:
        x.close()
    torch.cuda.empty_cache()
    return res


def prefill_section(pw, device, steps=5, warmup=2, tokens=0):
    """Mixtral-shaped prefill (4096 tokens, top-2 of 8 experts, H=4096,
    I=14336): the dequantise-to-shared-memory tcgen05 path."""
    import torch
    from any_precision_bitplane_gb300.layer import DeviceLayer
    from workloads import configs, gen
    cfg = configs.config_by_name("mixtral_prefill")
    T = tokens if tokens > 0 else cfg.T[0]
    layer = gen.make_layer(cfg, 0)
    dl = DeviceLayer(layer, device=device)
    tok = gen.make_tokens(layer, T)
    ids, wts = pw.route_topk(torch.from_numpy(tok.logits).to(device), cfg.k)
    hidden = torch.from_numpy(tok.hidden_bf16.view(np.int16)).to(device)
    out = torch.empty((T, cfg.H), dtype=torch.float32, device=device)
    ws = torch.empty(pw.workspace_bytes(T, cfg.H, cfg.I, cfg.E, cfg.k), dtype=torch.uint8,
                     device=device)
    for _ in range(warmup):
        pw.moe_forward(hidden, ids, wts, dl.table, cfg.I, cfg.E, out=out, workspace=ws)
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(steps):
        pw.moe_forward(hidden, ids, wts, dl.table, cfg.I, cfg.E, out=out, workspace=ws)
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / steps
    flops = 2.0 * T * cfg.k * (cfg.H * 2 * cfg.I + cfg.I * cfg.H)
    peak, kind = tensor_peak()
    tflops = flops / (ms / 1e3) / 1e12
    # the dominant kernel (gate_up dequant-GEMM), timed with events around its launches
    stream = torch.cuda.Stream(device)
    gu_ms = time_dominant(pw, cfg, [dl], hidden, ids, wts, steps, stream)
    gu_flops = 2.0 * T * cfg.k * cfg.H * 2 * cfg.I
    gu_tflops = gu_flops / (gu_ms / 1e3) / 1e12
    dl.close()
    del ws
    torch.cuda.empty_cache()
    return {"workload": "%s: H=%d I=%d E=%d top-%d, T=%d" % (cfg.name, cfg.H, cfg.I, cfg.E,
                                                            cfg.k, T),
            "tokens_per_s": T / (ms / 1e3), "ms_per_step": ms, "steps": steps,
            "roofline": {"bound": "tensor", "achieved": gu_tflops, "peak": peak,
                         "unit": "TFLOP/s", "frac": gu_tflops / peak, "peak_kind": kind,
                         "flops_per_launch": gu_flops, "ms_per_launch": gu_ms,
                         "kernel": "dq_gemm_kernel<gate_up> (dequant + tcgen05 GEMM + SiLU; "
                                   "the call's largest launch)",
                         "traffic": recorded_traffic("dq_gemm_kernel<0>", cfg.name, T)},
            "call_roofline": {"bound": "tensor", "achieved": tflops, "peak": peak,
                              "unit": "TFLOP/s", "frac": tflops / peak,
                              "flops_per_call": flops,
                              "kernel": "whole prefill call (permute, gather, gate_up and down "
                                        "dequant+tcgen05 GEMMs, combine)"}}


def native(args):
    import torch
    import any_precision_bitplane_gb300 as pw
    rank, world, local = dist_env()
    if args.prefill_only:
        torch.cuda.set_device(local)
        pw.lib()
        print(json.dumps(prefill_section(pw, torch.device("cuda", local), steps=args.steps,
                                         warmup=args.warmup, tokens=args.prefill_tokens)),
              flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    pw.lib()
    peak, peak_kind = measured_peaks()

    cfg, layer, layers, hidden, ids, wts, step_bytes, weight_bytes, host = \
        setup_workload(args.workload, args.T, device, args.copies, args.uniform_q)
    stream = torch.cuda.Stream(device)
    g, start, stop, out = time_device(pw, cfg, layers, hidden, ids, wts, args.steps,
                                      args.warmup, stream)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        g.replay()
        stop.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.2)
    sampler.stop()
    T = args.T
    ms = slowest_rank_seconds(start.elapsed_time(stop) / 1e3, world, device) * 1e3
    value = T * args.steps * world / (ms / 1e3)   # the slowest rank's time, all ranks' tokens
    per_launch_s = ms / 1e3 / args.steps
    achieved = step_bytes / per_launch_s / 1e9

    # dominant kernel (decode gate_up): its own launches timed with events
    dom_ms = time_dominant(pw, cfg, layers, hidden, ids, wts, args.steps, stream)
    ids_np = ids.cpu().numpy()
    gu_bytes = (layers[0].routed_bytes(ids_np, blocks=(0,)) + hidden_bytes(cfg, args.T) +
                args.T * cfg.k * cfg.I * 4)
    dom_achieved = gu_bytes / (dom_ms / 1e3) / 1e9

    e2e = None
    if not args.no_e2e:
        e2e_dt, bi, bo = time_e2e(pw, cfg, layers, host, args.steps, args.warmup, device)
        e2e = {"value": job_tokens_per_s(T * args.steps, e2e_dt, world, device),
               "unit": "tokens/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "mode": "C ABI with pinned host buffers read/written by the kernels, K steps "
                       "in one CUDA graph, wall clock"}

    sweep = {}
    if not args.no_sweep and rank == 0 and world == 1:
        for t2 in cfg.T:
            if t2 == T:
                continue
            c2, _, l2, hd2, id2, w2, sb2, _, _ = setup_workload(args.workload, t2, device)
            g2, s2, e2, _ = time_device(pw, c2, l2, hd2, id2, w2, args.steps, args.warmup, stream)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                s2.record(stream)
                g2.replay()
                e2.record(stream)
            torch.cuda.synchronize()
            ms2 = s2.elapsed_time(e2)
            gbs = sb2 / (ms2 / 1e3 / args.steps) / 1e9
            sweep["T=%d" % t2] = {"tokens_per_s": t2 * args.steps / (ms2 / 1e3),
                                  "us_per_step": ms2 * 1e3 / args.steps,
                                  "GB_per_s": gbs, "frac": gbs / peak,
                                  "bytes_per_step": sb2}
            for x in l2:
                x.close()
            del g2
            torch.cuda.empty_cache()

    prefill = None
    configs_out = {}
    if not args.no_sweep and rank == 0 and world == 1:
        configs_out["mixtral_decode T=4"] = decode_config(pw, "mixtral_decode", 4, device, stream,
                                                          args.steps, args.warmup)
        configs_out["qwen3_decode T=64"] = decode_config(pw, "qwen3_decode", 64, device, stream,
                                                         args.steps, args.warmup, recommit=True)
        prefill = prefill_section(pw, device)

    clocks = sampler.summary(w0, w1)
    line = {
        "metric": metric_name(cfg.name),
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp32 accumulate (bf16 activations, 3-8 bit LUT weights)",
        "data": "synthetic (seeded codes, LUTs, bitwidths, hidden states and router logits)",
        "config": {"workload": "%s: H=%d I=%d E=%d top-%d, T=%d tokens per step" %
                               (cfg.name, cfg.H, cfg.I, cfg.E, cfg.k, T),
                   "bitwidths": ("every block at q = %d" % args.uniform_q if args.uniform_q
                                 else "q drawn per block from {3,4,5,6,8}"),
                   "l2": ("inputs larger than L2: " if len(layers) * weight_bytes > L2_BYTES
                          else "inputs fit in L2 (not HBM-bound): ") +
                         "%d rotating layer copies, %.1f MB of routed weights per step" %
                         (len(layers), weight_bytes / 1e6),
                   "timing": "CUDA events around one CUDA-graph replay of exactly K steps",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": dom_achieved, "peak": peak, "unit": "GB/s",
                     "frac": dom_achieved / peak, "peak_kind": peak_kind,
                     "kernel": "decode_gateup_kernel (gate_up + SiLU; the call's largest launch)",
                     "bytes_per_launch": gu_bytes, "ms_per_launch": dom_ms,
                     # the recorded counters are of the workload's own bitwidth mix
                     "traffic": (None if args.uniform_q else
                                 recorded_traffic("decode_gateup_kernel", args.workload, T))},
        "call_roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                          "frac": achieved / peak,
                          "kernel": "whole pw_moe_forward decode call (prep, gate_up, down "
                                    "+ combine)",
                          "bytes_per_call": step_bytes},
        "e2e": e2e,
        "gpu_launches": launches_per_call(cfg, T) * args.steps,
        "clocks": clocks,
    }
    if sweep:
        line["sweep"] = sweep
    if configs_out:
        line["configs"] = configs_out
    if prefill is not None:
        line["prefill"] = prefill
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, T)
    if rank == 0:
        print(json.dumps(line), flush=True)
    for x in layers:
        x.close()
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- reference arm

def reference(args):
    """The CPU oracle on the same workload and metric.  One step = one routed
    (token, expert) pair of the batch through the oracle (1/k of a token), so
    that any --steps stays a bounded amount of CPU work."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import moe
    cfg, tok, ids, w, block = _oracle_setup(args.workload, args.T)
    T, k = ids.shape

    def step(i):
        t, j = (i // k) % T, i % k
        y = moe.expert_outputs(tok.hidden_bf16, ids, block, cfg.E, experts=[int(ids[t, j])],
                               tokens=[t])
        return float(w[t, j]) * y[t * k + j]

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = (args.steps / k) / dt
    print(json.dumps({
        "impl": "reference",
        "metric": metric_name(cfg.name),
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "%s: H=%d I=%d E=%d top-%d, T=%d tokens per step" %
                               (cfg.name, cfg.H, cfg.I, cfg.E, cfg.k, args.T)},
        "cpu_baseline": dict({"value": value, "unit": "tokens/s", "kind": "oracle",
                              "sample": "each step: one routed (token, expert) pair of the "
                                        "batch through the oracle, i.e. 1/%d of a token" % k},
                             **host_cores_entry()),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
