#!/usr/bin/env python
"""Benchmark of the MoE expert-layer forward (route -> permute -> grouped
SwiGLU FFN -> combine) through libmoe's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one whole-layer forward over the workload's batch of T tokens
(all four steps of the layer).  The default workload is the largest
single-GPU one, `fine_grained` (T=8192, H=7168, F=2048, E=256, k=8).  Prints
ONE JSON line (rank 0): the value and the kernel breakdown of that workload,
`configs` with every other workload of record measured in the same process,
and `protocol` with the median and spread of the time per step over three
input realizations in this process and in a fresh one.  Under torchrun every
rank runs the same workload on its own GPU with no data-path collective
(independent replicas, weak scaling); `value` is the tokens of all ranks
divided by the slowest rank's time.

`--impl reference` times the CPU oracle (fp64, the machine's host cores) on a
bounded sample of the same workload.
"""
from __future__ import annotations

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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routing_grouped_expert_gb300 import accounting as acc  # noqa: E402
from routing_grouped_expert_gb300 import inputs as I  # noqa: E402

METRIC = "MoE-layer tokens/s; grouped-GEMM % of bf16 TC peak or % HBM GB/s roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 10**6
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ setup
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="fine_grained", choices=sorted(I.WORKLOADS))
    ap.add_argument("--shape", default=None,
                    help="T,H,F,E,k: a uniform-routing workload of these sizes instead")
    ap.add_argument("--sweep", action="store_true",
                    help="tokens-per-expert sweep of the workload's shape (own JSON line)")
    ap.add_argument("--train", action="store_true",
                    help="time a training step: moe_forward_train + moe_backward (own JSON line)")
    ap.add_argument("--gated", action="store_true",
                    help="time the layer from hidden states (router projection + routed "
                         "experts + --shared-f shared expert) instead (own JSON line)")
    ap.add_argument("--shard-f", action="store_true",
                    help="time the layer split over the ranks along the FFN features: each "
                         "rank's fp32 partial, one all-reduce, one rounding (own JSON line)")
    ap.add_argument("--shared-f", type=int, default=0,
                    help="FFN width of the shared expert for --gated (0 = none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads of record (the `configs` key)")
    ap.add_argument("--no-protocol", action="store_true",
                    help="skip the median over realizations and processes (`protocol` key)")
    ap.add_argument("--protocol-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.shape:
        T, H, F, E, k = (int(v) for v in args.shape.split(","))
        name = f"shape_T{T}_H{H}_F{F}_E{E}_k{k}"
        I.WORKLOADS[name] = I.small(name, T=T, H=H, F=F, E=E, k=k)
        args.workload = name
    return args


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu
    record, or None when there is none or the kernel's sources changed since
    the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[f"{workload}:{kernel}"]
        blob = b"".join(open(os.path.join(ROOT, p), "rb").read() for p in rec["sources"])
    except (OSError, KeyError, ValueError):
        return None
    if hashlib.sha256(blob).hexdigest() != rec["source_sha256"]:
        return None
    return int(rec["bytes_per_launch"])


def wl_config(wl, extra=None):
    cfg = {"workload": wl.name, "T": wl.T, "H": wl.H, "F": wl.F, "E": wl.E, "k": wl.k,
           "routing": "uniform" if wl.skew_alpha == 0 else
           f"zipf(s={wl.zipf_s}) bias, alpha={wl.skew_alpha}",
           "inputs": "x~N(0,1) bf16, W1/W3~N(0,1/H), W2~N(0,1/F) bf16, logits~N(0,1) fp32, "
                     "seeded"}
    if extra:
        cfg.update(extra)
    return cfg


# ------------------------------------------------- multi-rank aggregation
def max_over_ranks(v: float, world: int, device) -> float:
    """The slowest rank's time (all ranks must call this)."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(world: int, T: int, K: int, region_ms: float) -> float:
    """Whole-job tokens/s: every rank processes T tokens per step."""
    return world * T * K / (region_ms / 1e3)


# --------------------------------------------------------- clock sampling
class ClockSampler:
    """nvidia-smi samples every 100 ms, stamped on arrival; keeps those that
    fall inside [begin, end]."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.begin = self.end = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_begin(self):
        self.begin = time.time()

    def mark_end(self):
        self.end = time.time()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.begin - 0.05 <= r[0] <= self.end + 0.15]
        if not inside and rows:   # timed region shorter than one sample period
            mid = 0.5 * (self.begin + self.end)
            inside = [min(rows, key=lambda r: abs(r[0] - mid))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for _, p in inside if num(p[0]) is not None]
        smax = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in inside:
            for n, v in zip(names, p[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        power = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ our kernels
OTHER_CONFIGS = ("tiny", "mixtral_decode", "dbrx_prefill", "fine_grained", "skewed",
                 "skewed_10x")


class Inputs:
    """Inputs of the workloads measured in one run.  Workloads of the same
    shape and realization share one copy of the weights (the seeds depend on
    nothing else), so the skewed workloads reuse the fine-grained weights."""

    def __init__(self, dev):
        self.dev = dev
        self.weights = {}

    def get(self, wl):
        key = (wl.H, wl.F, wl.E, wl.realization)
        if key not in self.weights:
            self.weights = {k: v for k, v in self.weights.items() if k[3] == 0}
            torch.cuda.empty_cache()
            self.weights[key] = I.make_weights(wl, self.dev)
        W1, W3, W2 = self.weights[key]
        return dict(x=I.make_x(wl, self.dev), logits=I.make_logits(wl).to(self.dev),
                    W1=W1, W3=W3, W2=W2)


def routing_stats(moe, wl, d, ws):
    idx, _ = moe.moe_route_topk(d["logits"], wl.k, ws=ws)
    counts = moe.moe_permute(idx, wl.E, ws=ws)[0].cpu()
    return int((counts > 0).sum()), int(counts.max())


def time_forward(moe, wl, d, ws, K, warmup, world, dev, sample_clocks, local=0):
    """K plain moe_forward steps after `warmup` untimed ones.  With weights that
    fit in L2 the L2 is flushed before every step and each step is bracketed
    by its own events, so the flush is not counted.  Returns (ms per step over
    the slowest rank, clocks summary or None, flush)."""
    touched, _ = routing_stats(moe, wl, d, ws)
    flush = acc.expert_weight_bytes(wl.H, wl.F, touched) < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    args = (d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
    for _ in range(warmup):
        moe.moe_forward(*args, out=out, ws=ws)
    st = moe.moe_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {moe.moe_status_string(st)}")
    step_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if sample_clocks else None
    barrier()
    if clocks:
        time.sleep(0.3)
        clocks.mark_begin()
    t_start.record()
    for i in range(K):
        if flush:
            flush_buf.zero_()
            step_evs[i][0].record()
        moe.moe_forward(*args, out=out, ws=ws)
        if flush:
            step_evs[i][1].record()
    t_end.record()
    barrier()
    if clocks:
        clocks.mark_end()
    st = moe.moe_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {moe.moe_status_string(st)}")
    region_ms = (sum(e[0].elapsed_time(e[1]) for e in step_evs) if flush
                 else t_start.elapsed_time(t_end))
    region_ms = max_over_ranks(region_ms, world, dev)
    return region_ms / K, (clocks.summary() if clocks else None), flush


def time_graph(moe, wl, d, K, warmup, dev, flush):
    """K launches of the layer captured once as a CUDA graph (moe.ForwardGraph,
    its own workspace), on a side stream, under the same L2 rule as
    time_forward (flushed before every step and each step between its own
    events when the weights fit in L2).  Returns ms per step."""
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        g = moe.ForwardGraph(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k, out=out)
        for _ in range(warmup):
            g.launch()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        s.synchronize()
        t0.record()
        for i in range(K):
            if flush:
                flush_buf.zero_()
                evs[i][0].record()
            g.launch()
            if flush:
                evs[i][1].record()
        t1.record()
        s.synchronize()
        st = moe.moe_get_device_status(g.ws)
        g.close()
    torch.cuda.current_stream(dev).wait_stream(s)
    if st != 0:
        raise RuntimeError(f"device status after graph launches: {moe.moe_status_string(st)}")
    region = sum(e[0].elapsed_time(e[1]) for e in evs) if flush else t0.elapsed_time(t1)
    return region / K


def time_stages(moe, wl, d, ws, K, dev, flush):
    """K moe_forward_events steps: each kernel's mean duration, from one CUDA
    event between consecutive kernels on the launch stream."""
    nst = moe.FORWARD_STAGES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(K)]
    torch.cuda.synchronize(dev)
    for i in range(K):
        if flush:
            flush_buf.zero_()
        moe.moe_forward_events(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k, evs[i],
                               out=out, ws=ws)
    torch.cuda.synchronize(dev)
    names = [moe.moe_forward_stage_name(j) for j in range(nst)]
    mean_ms = {n: statistics.fmean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
               for j, n in enumerate(names)}
    per_step = statistics.fmean(evs[i][0].elapsed_time(evs[i][nst]) for i in range(K))
    return mean_ms, per_step


def kernel_roofline(wl, mean_ms, touched, peaks, peak_src, kernel=None):
    """The roofline of one kernel (the dominant one unless named): algorithmic
    bytes or FLOPs of a launch over its mean duration, against the measured
    copy bandwidth or the sustained bf16 rate, whichever bounds it."""
    P = wl.T * wl.k
    top = kernel or max(mean_ms, key=mean_ms.get)
    kbytes = {"route": acc.route_bytes(wl.T, wl.E, wl.k),
              "scan": 0, "scatter": 4 * P * 4,
              "gather": 0 if acc.ffn_gathers_rows(wl.T, wl.k, wl.E) else
              acc.gather_bytes(wl.T, wl.k, wl.H),
              "fc1": acc.fc1_bytes(wl.H, wl.F, touched, wl.T, wl.k, wl.E),
              "fc2": acc.fc2_bytes(wl.H, wl.F, touched, P),
              "combine": acc.combine_bytes(wl.T, wl.H, wl.k)}
    kflops = {"fc1": 2 * P * wl.H * 2 * wl.F, "fc2": 2 * P * wl.F * wl.H}
    sec = mean_ms[top] / 1e3
    tflops_peak = peaks["bf16_tflops_sustained"]
    t_mem = kbytes.get(top, 0) / (peaks["hbm_gbs"] * 1e9)
    t_tc = kflops.get(top, 0) / (tflops_peak * 1e12)
    if t_tc > t_mem:
        achieved = kflops[top] / sec / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tflops_peak,
                "unit": "TFLOP/s", "frac": round(achieved / tflops_peak, 4)}
        peak_note = f"bf16_tflops_sustained ({peak_src})"
    else:
        achieved = kbytes.get(top, 0) / sec / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
        peak_note = f"hbm_gbs ({peak_src})"
    roof.update({"traffic": measured_traffic(wl.name, top), "kernel": top,
                 "algorithmic_bytes": kbytes.get(top), "algorithmic_flops": kflops.get(top),
                 "kernel_ms": round(mean_ms[top], 5), "peak_source": peak_note})
    if roof["frac"] > 1.0:
        roof["above_peak"] = ("the denominator is a measured copy (read + write streams); a "
                              "read-dominated kernel can run above it")
    return roof


def layer_roofline(wl, ms_per_step, touched, peaks):
    flops = acc.ffn_flops(wl.T, wl.H, wl.F, wl.k)
    lbytes = acc.layer_bytes(wl.T, wl.H, wl.F, wl.E, wl.k, touched)
    t_roof, bound = acc.roofline_seconds(flops, lbytes, peaks["bf16_tflops"] * 1e12,
                                         peaks["hbm_gbs"] * 1e9)
    return {"flops": flops, "bytes": lbytes, "t_roof_ms": round(t_roof * 1e3, 4),
            "bound": bound, "frac": round(t_roof / (ms_per_step / 1e3), 4),
            "tflops": round(flops / (ms_per_step / 1e3) / 1e12, 2),
            "hbm_gbs": round(lbytes / (ms_per_step / 1e3) / 1e9, 1)}


def bench_ours(args, rank, world, local):
    import routing_grouped_expert_gb300 as moe

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[args.workload]
    pool = Inputs(dev)
    d = pool.get(wl)
    ws = moe.Workspace(dev)
    touched, max_count = routing_stats(moe, wl, d, ws)
    weight_bytes = acc.expert_weight_bytes(wl.H, wl.F, touched)
    P = wl.T * wl.k
    K = args.steps

    # the value: K plain moe_forward steps
    ms_per_step, clocks, flush = time_forward(moe, wl, d, ws, K, args.warmup, world, dev,
                                              rank == 0, local)
    value = throughput(world, wl.T, K, ms_per_step * K)
    # the per-kernel breakdown: a second region with stage events
    mean_ms, events_ms_per_step = time_stages(moe, wl, d, ws, K, dev, flush)
    # the same layer captured once as a CUDA graph and replayed (no host launches)
    graph_ms = time_graph(moe, wl, d, K, args.warmup, dev, flush) if world == 1 else None

    # end to end: host activations in, host result out, through the C ABI
    e2e = None
    if not args.no_e2e:
        xh = d["x"].cpu().pin_memory()
        lh = d["logits"].cpu().pin_memory()
        oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        flush_buf = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
                     if flush else None)
        for _ in range(max(3, args.warmup // 2)):
            moe.moe_forward_host(xh, lh, d["W1"], d["W3"], d["W2"], wl.k, out_host=oh, ws=ws)
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            if flush:
                flush_buf.zero_()
            moe.moe_forward_host(xh, lh, d["W1"], d["W3"], d["W2"], wl.k, out_host=oh, ws=ws)
        e1.record()
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": throughput(world, wl.T, K, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": wl.T * wl.H * 2 + wl.T * wl.E * 4,
               "d2h_bytes_per_step": wl.T * wl.H * 2,
               "ms_per_step": e2e_ms / K,
               "note": "moe_forward_host on pinned host buffers: x and the logits are read and "
                       "the result written across the host link by the kernels (each byte "
                       "once), inside the timed region" + (", L2 flushed between steps"
                                                           if flush else "")}

    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    kern_sum = sum(mean_ms.values())
    kernels = {n: {"ms": round(v, 5), "share": round(v / kern_sum, 4)} for n, v in mean_ms.items()}
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": wl_config(wl, {
            "parallelism": f"replicas x{world} (no collective)" if world > 1 else "single GPU",
            "l2": ("flushed between steps (inputs fit in L2)" if flush else
                   f"inputs larger than L2 ({weight_bytes / 1e9:.2f} GB of expert weights "
                   f"streamed per step)"),
            "touched_experts": touched, "max_expert_count": max_count,
            "mean_expert_count": P / wl.E}),
        "roofline": kernel_roofline(wl, mean_ms, touched, peaks, peak_src),
        "layer_roofline": layer_roofline(wl, ms_per_step, touched, peaks),
        "kernels": kernels,
        "kernels_timing": ("per-stage CUDA events on the launch stream, in a second timed "
                           f"region of {K} moe_forward_events steps "
                           f"({events_ms_per_step:.4f} ms per step with the events)"),
        "gpu_launches": acc.forward_launches(wl.T, wl.k, wl.E) * K,
        "clocks": clocks,
    }
    if e2e:
        result["e2e"] = e2e
    if graph_ms is not None:
        result["graph"] = {"ms_per_step": round(graph_ms, 5),
                           "value": round(wl.T / graph_ms * 1e3, 1), "unit": UNIT,
                           "how": "moe.ForwardGraph: the layer captured once as a CUDA graph, "
                                  f"{K} launches, same L2 rule as the value"}
    if world == 1 and not args.no_configs:
        result["configs"] = bench_configs(moe, args, pool, ws, dev, wl.name, ms_per_step)
    if world == 1 and not args.no_protocol:
        result["protocol"] = bench_protocol(moe, args, pool, ws, dev, wl, ms_per_step)
    return result, d


def bench_configs(moe, args, pool, ws, dev, main_name, main_ms):
    """Every other workload of record, measured in this process: time per
    step, the layer's roofline fraction, the dominant kernel's roofline and
    the clocks of its timed region; the skewed workloads also as a ratio to
    the uniform fine-grained time."""
    peaks, peak_src = load_peaks()
    out = {}
    times = {main_name: main_ms}
    for name in OTHER_CONFIGS:
        if name == main_name:
            continue
        wl = I.WORKLOADS[name]
        d = pool.get(wl)
        touched, max_count = routing_stats(moe, wl, d, ws)
        K = max(10, args.steps)
        ms, clocks, flush = time_forward(moe, wl, d, ws, K, max(3, args.warmup), 1, dev, True)
        mean_ms, _ = time_stages(moe, wl, d, ws, K, dev, flush)
        graph_ms = time_graph(moe, wl, d, K, max(3, args.warmup), dev, flush)
        times[name] = ms
        lay = layer_roofline(wl, ms, touched, peaks)
        roof = kernel_roofline(wl, mean_ms, touched, peaks, peak_src)
        out[name] = {"T": wl.T, "H": wl.H, "F": wl.F, "E": wl.E, "k": wl.k,
                     "ms_per_step": round(ms, 5), "tokens_per_s": round(wl.T / ms * 1e3, 1),
                     "layer_frac": lay["frac"], "layer_bound": lay["bound"],
                     "layer_tflops": lay["tflops"],
                     "kernel": roof["kernel"], "kernel_frac": roof["frac"],
                     "kernel_bound": roof["bound"], "kernel_ms": roof["kernel_ms"],
                     "touched_experts": touched, "max_expert_count": max_count,
                     "l2": "flushed between steps" if flush else "inputs larger than L2",
                     "graph_ms_per_step": round(graph_ms, 5),
                     "graph_layer_frac": layer_roofline(wl, graph_ms, touched, peaks)["frac"],
                     "steps": K, "clocks": clocks}
        del d
    if "fine_grained" in times:
        for name in ("skewed", "skewed_10x"):
            if name in out:
                out[name]["ratio_to_fine_grained"] = round(times[name] / times["fine_grained"], 4)
    return out


def bench_protocol(moe, args, pool, ws, dev, wl, main_ms):
    """The headline as a median: the workload's time per step on three
    realizations of its inputs (seeds shifted by 1000 r), measured here and in a
    second, fresh process; reports the median and the spread of the six."""
    K = max(10, args.steps)
    here = []
    for r in range(3):
        w = wl.with_(realization=r)
        d = pool.get(w)
        ms, _, _ = time_forward(moe, w, d, ws, K, max(3, args.warmup), 1, dev, False)
        here.append(ms)
        del d
    pool.weights = {k: v for k, v in pool.weights.items() if k[3] == 0}
    torch.cuda.empty_cache()
    cmd = [sys.executable, os.path.abspath(__file__), "--protocol-child", "--workload", wl.name,
           "--steps", str(K), "--warmup", str(max(3, args.warmup))]
    there = []
    try:
        res = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
        there = json.loads(res.stdout.strip().splitlines()[-1])["ms"] if res.returncode == 0 else []
    except (subprocess.TimeoutExpired, ValueError, IndexError, KeyError):
        there = []
    allv = here + there
    return {"ms_per_step_median": round(statistics.median(allv), 5),
            "ms_per_step_min": round(min(allv), 5), "ms_per_step_max": round(max(allv), 5),
            "spread": round((max(allv) - min(allv)) / statistics.median(allv), 4),
            "this_process_ms": [round(v, 5) for v in here],
            "fresh_process_ms": [round(v, 5) for v in there],
            "how": f"{K} timed steps per realization; realizations r = 0, 1, 2 (seeds + 1000 r) "
                   "in this process and again in a fresh process"}


def protocol_child(args):
    import routing_grouped_expert_gb300 as moe
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[args.workload]
    pool = Inputs(dev)
    ws = moe.Workspace(dev)
    ms = []
    for r in range(3):
        w = wl.with_(realization=r)
        d = pool.get(w)
        ms.append(time_forward(moe, w, d, ws, args.steps, args.warmup, 1, dev, False)[0])
        del d
    print(json.dumps({"ms": ms}), flush=True)


# ------------------------------------------------------- the CPU oracle
class _ExpertCache(dict):
    """W[e] -> the expert's matrix as an exact fp64 host array, copied once."""

    def __init__(self, W):
        super().__init__()
        self.W = W

    def __missing__(self, e):
        a = self.W[e].to("cpu", torch.float64).numpy()
        self[e] = a
        return a


def oracle_sampler(wl, d, mem_cap=12 * 2**30, max_pool=64):
    """A pool of the batch's first tokens whose experts' fp64 weights fit in
    `mem_cap`, and a function that runs the oracle on n of them."""
    from oracle import moe_oracle as O
    logits = d["logits"].cpu()
    idx, _ = O.route_topk(logits.numpy(), wl.k)
    per_expert = acc.expert_weight_bytes(wl.H, wl.F, 1, elem=8)
    pool, experts = [], set()
    for t in range(wl.T):
        new = experts | set(idx[t].tolist())
        if pool and (len(new) * per_expert > mem_cap or len(pool) >= max_pool):
            break
        pool.append(t)
        experts = new
    x_pool = d["x"][torch.tensor(pool, device=d["x"].device)].cpu()
    l_pool = logits[pool]
    W1c, W3c, W2c = _ExpertCache(d["W1"]), _ExpertCache(d["W3"]), _ExpertCache(d["W2"])
    for e in sorted(experts):                 # copy outside any timed region
        W1c[e], W3c[e], W2c[e]
    state = {"next": 0}

    def run(n):
        n = max(1, min(n, len(pool)))
        s = state["next"]
        rows = [(s + i) % len(pool) for i in range(n)]
        state["next"] = (s + n) % len(pool)
        O.forward_perm(x_pool[rows], l_pool[rows].numpy(), W1c, W3c, W2c, wl.k)
        return n

    desc = (f"oracle forward_perm on sub-batches drawn from the first {len(pool)} tokens "
            f"(their {len(experts)} experts' weights pre-copied as exact fp64)")
    return run, desc


def cpu_baseline(wl, d, seconds=10.0):
    run, desc = oracle_sampler(wl, d)
    t0 = time.perf_counter()
    run(1)
    t1 = (time.perf_counter() - t0)
    n = max(1, min(32, int(1.0 / max(t1, 1e-6))))
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        done += run(n)
    el = time.perf_counter() - t0
    return {"value": round(done / el, 3), "unit": UNIT, "cores": torch.get_num_threads(),
            "kind": "oracle", "sample": f"{done} tokens in {el:.1f} s; {desc}; "
                                       f"sub-batches of {n} tokens"}


def bench_reference(args, rank, world, local):
    if rank != 0:
        return None
    wl = I.WORKLOADS[args.workload]
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    d = I.make_inputs(wl, dev)
    run, desc = oracle_sampler(wl, d)
    budget = 150.0 / max(1, args.steps + args.warmup)   # seconds per step
    t0 = time.perf_counter()
    run(1)
    t1 = time.perf_counter() - t0
    n = max(1, min(32, int(budget / max(t1, 1e-6))))
    for _ in range(args.warmup):
        run(n)
    done, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        done += run(n)
    el = time.perf_counter() - t0
    value = done / el
    cb = {"value": round(value, 3), "unit": UNIT, "cores": torch.get_num_threads(),
          "kind": "oracle", "sample": f"{n} tokens per step; {desc}"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wl_config(wl, {"parallelism": "host CPU (rank 0)"}),
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------ tokens-per-expert sweep
def bench_sweep(args):
    """Expert-layer time against tokens per expert b_e = T*k/E for the
    workload's (H, F, E, k), with a least-squares fit of the linear expert
    time model Te = k3 * b_e + k4 ("MegaScale-Infer", §3.4 Performance
    Simulation Model) and the utilisation model util = min(k/E * B/F * b, 1)
    ("MegaScale-Infer", §2) evaluated with the measured peaks."""
    import routing_grouped_expert_gb300 as moe
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    base = I.WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    W1, W3, W2 = I.make_weights(base, dev)
    ws = moe.Workspace(dev)
    nst = moe.FORWARD_STAGES
    points = []
    for be in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048):
        T = max(1, be * base.E // base.k)
        wl = base.with_(T=T, name=f"{base.name}_be{be}")
        x = I.make_x(wl, dev)
        logits = I.make_logits(wl).to(dev)
        out = torch.empty(T, base.H, dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            moe.moe_forward(x, logits, W1, W3, W2, base.k, out=out, ws=ws)
        K = max(5, min(args.steps, 50))
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(K)]
        torch.cuda.synchronize(dev)
        for i in range(K):
            moe.moe_forward_events(x, logits, W1, W3, W2, base.k, evs[i], out=out, ws=ws)
        torch.cuda.synchronize(dev)
        if moe.moe_get_device_status(ws) != 0:
            raise RuntimeError("device status after sweep point")
        names = [moe.moe_forward_stage_name(j) for j in range(nst)]
        f1, f2 = names.index("fc1"), names.index("fc2") + 1
        step = statistics.median(evs[i][0].elapsed_time(evs[i][nst]) for i in range(K))
        ffn = statistics.median(evs[i][f1].elapsed_time(evs[i][f2]) for i in range(K))
        flops = acc.ffn_flops(T, base.H, base.F, base.k)
        util = acc.util(base.k, base.E, peaks["hbm_gbs"] * 1e9, peaks["bf16_tflops"] * 1e12, T)
        points.append({"tokens_per_expert": be, "T": T, "layer_ms": round(step, 5),
                       "ffn_ms": round(ffn, 5), "ffn_tflops": round(flops / ffn / 1e9, 2),
                       "ffn_frac_of_peak": round(flops / ffn / 1e9 / peaks["bf16_tflops"], 4),
                       "util_model": round(util, 4)})
    # least squares Te = k3 * b_e + k4 on the FFN time
    xs = [p["tokens_per_expert"] for p in points]
    ys = [p["ffn_ms"] * 1e3 for p in points]
    n = len(xs)
    mx, my = sum(xs) / n, sum(ys) / n
    sxx = sum((a - mx) ** 2 for a in xs)
    sxy = sum((a - mx) * (b - my) for a, b in zip(xs, ys))
    k3 = sxy / sxx
    k4 = my - k3 * mx
    ss_res = sum((b - (k3 * a + k4)) ** 2 for a, b in zip(xs, ys))
    ss_tot = sum((b - my) ** 2 for b in ys)
    ridge = acc.ridge_tokens(peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9)
    return {"sweep": "tokens_per_expert", "shape": {"H": base.H, "F": base.F, "E": base.E,
                                                    "k": base.k},
            "peaks": {**peaks, "source": peak_src},
            "ridge_tokens_per_expert": round(ridge * base.k / base.E, 1),
            "fit_Te_us": {"k3_us_per_token": round(k3, 4), "k4_us": round(k4, 2),
                          "r2": round(1 - ss_res / ss_tot, 5)},
            "points": points}


# ----------------------------------------------- layer from hidden states
def bench_gated(args):
    """moe_forward_gated: router projection x @ Wg, the routed layer, and an
    optional shared expert of width --shared-f added to every token."""
    import routing_grouped_expert_gb300 as moe
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[args.workload]
    d = I.make_inputs(wl, dev)
    g = torch.Generator(device=dev).manual_seed(6)
    Wg = (torch.randn(wl.H, wl.E, generator=g, device=dev) / math.sqrt(wl.H)).to(torch.bfloat16)
    Fs = args.shared_f
    shared = None
    if Fs:
        shared = tuple((torch.randn(r, c, generator=g, device=dev) / math.sqrt(r)).to(
            torch.bfloat16) for r, c in ((wl.H, Fs), (wl.H, Fs), (Fs, wl.H)))
    ws = moe.Workspace(dev)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    run = lambda: moe.moe_forward_gated(d["x"], Wg, d["W1"], d["W3"], d["W2"], wl.k,  # noqa
                                        shared=shared, out=out, ws=ws)
    for _ in range(args.warmup):
        run()
    if moe.moe_get_device_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    peaks, peak_src = load_peaks()
    idx = moe.moe_route_topk(moe.moe_router_logits(d["x"], Wg), wl.k)[0]
    touched = int((moe.moe_permute(idx, wl.E)[0] > 0).sum())
    flops = acc.ffn_flops(wl.T, wl.H, wl.F, wl.k) + 2 * wl.T * wl.H * wl.E \
        + 2 * wl.T * 3 * wl.H * Fs
    nbytes = acc.layer_bytes(wl.T, wl.H, wl.F, wl.E, wl.k, touched) + wl.H * wl.E * 2 \
        + 3 * wl.H * Fs * 2
    t_roof, bound = acc.roofline_seconds(flops, nbytes, peaks["bf16_tflops"] * 1e12,
                                         peaks["hbm_gbs"] * 1e9)
    return {"metric": METRIC, "mode": "gated", "value": round(wl.T / (ms / 1e3), 1),
            "unit": UNIT, "ms_per_step": round(ms, 5), "steps": args.steps,
            "config": wl_config(wl, {"router": f"x @ Wg [{wl.H}, {wl.E}] bf16 -> fp32",
                                     "shared_expert_F": Fs, "touched_experts": touched}),
            "layer_roofline": {"flops": flops, "bytes": nbytes, "t_roof_ms": round(t_roof * 1e3, 4),
                               "bound": bound, "frac": round(t_roof / (ms / 1e3), 4),
                               "tflops": round(flops / (ms / 1e3) / 1e12, 2),
                               "peak_source": peak_src}}


# ------------------------------------------------- feature-sharded layer
def bench_shard(args, rank, world, local):
    """The layer split over `world` ranks along the FFN features: every rank
    routes all T tokens and computes its slice's fp32 partial output; one
    all-reduce sums them and the sum is rounded once.  Strong scaling: the
    job's work per step is one layer of T tokens whatever the rank count."""
    import routing_grouped_expert_gb300 as moe
    from routing_grouped_expert_gb300 import sharded
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[args.workload]
    W1, W3, W2 = I.make_weights(wl, dev)
    W1s, W3s, W2s = sharded.shard_weights(W1, W3, W2, world, rank)
    del W1, W3, W2
    torch.cuda.empty_cache()
    x, logits = I.make_x(wl, dev), I.make_logits(wl).to(dev)
    ws = moe.Workspace(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        sharded.sharded_forward(x, logits, W1s, W3s, W2s, wl.k, ws=ws)
    if moe.moe_get_device_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record()
    for _ in range(args.steps):
        sharded.sharded_forward(x, logits, W1s, W3s, W2s, wl.k, ws=ws)
    e1.record()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    if rank != 0:
        return None
    return {"metric": METRIC, "mode": "shard_f", "value": round(wl.T / (ms / 1e3), 1),
            "unit": UNIT, "n_gpus": world, "ms_per_step": round(ms, 5), "steps": args.steps,
            "warmup": args.warmup, "scaling": "strong", "dtype": "bf16", "data": "synthetic",
            "config": wl_config(wl, {"parallelism": f"FFN features split over {world} "
                                                    f"rank(s), one fp32 all-reduce",
                                     "F_per_rank": W1s.shape[2]})}


# --------------------------------------------------------- training step
def bench_train(args):
    """moe_forward_train then moe_backward on the workload, dout ~ N(0, 1).
    FLOPs: forward 2*T*k*3*H*F, backward twice that (DGrad and WGrad)."""
    import routing_grouped_expert_gb300 as moe
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[args.workload]
    d = I.make_inputs(wl, dev)
    g = torch.Generator(device=dev).manual_seed(7)
    dout = torch.randn(wl.T, wl.H, generator=g, device=dev).to(torch.bfloat16)
    ws = moe.Workspace(dev)

    def step(ev=None):
        if ev:
            ev[0].record()
        moe.moe_forward_train(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k, ws)
        if ev:
            ev[1].record()
        r = moe.moe_backward(dout, d["logits"], d["W1"], d["W3"], d["W2"], wl.k, ws)
        if ev:
            ev[2].record()
        return r
    for _ in range(args.warmup):
        step()
    if moe.moe_get_device_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize(dev)
    fwd = statistics.fmean(e[0].elapsed_time(e[1]) for e in evs)
    bwd = statistics.fmean(e[1].elapsed_time(e[2]) for e in evs)
    ms = fwd + bwd
    peaks, peak_src = load_peaks()
    f_flops = acc.ffn_flops(wl.T, wl.H, wl.F, wl.k)
    flops = 3 * f_flops
    return {"metric": METRIC, "mode": "train", "value": round(wl.T / (ms / 1e3), 1), "unit": UNIT,
            "ms_per_step": round(ms, 4), "forward_ms": round(fwd, 4), "backward_ms": round(bwd, 4),
            "steps": args.steps, "config": wl_config(wl, {"dout": "N(0,1) bf16"}),
            "tflops": round(flops / (ms / 1e3) / 1e12, 1),
            "backward_tflops": round(2 * f_flops / (bwd / 1e3) / 1e12, 1),
            "frac_of_bf16_peak": round(flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
            "peak_source": peak_src}


def main():
    args = parse()
    if args.protocol_child:
        protocol_child(args)
        return
    if args.train:
        print(json.dumps(bench_train(args)), flush=True)
        return
    if args.gated:
        print(json.dumps(bench_gated(args)), flush=True)
        return
    if args.sweep:
        print(json.dumps(bench_sweep(args)), flush=True)
        return
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.shard_f:
        res = bench_shard(args, rank, world, local)
        if res is not None:
            print(json.dumps(res), flush=True)
    elif args.impl == "reference":
        res = bench_reference(args, rank, world, local)
        if res is not None:
            print(json.dumps(res), flush=True)
    else:
        out = bench_ours(args, rank, world, local)
        if out is not None:
            res, d = out
            if world == 1 and not args.no_cpu_baseline:
                wl = I.WORKLOADS[args.workload]
                res["cpu_baseline"] = cpu_baseline(wl, d)
            print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
