#!/usr/bin/env python
"""Benchmark of the MoE expert-layer forward (route -> permute -> grouped
SwiGLU FFN -> combine) through libmoe's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one whole-layer forward over the workload's batch of T tokens
(all four steps of the layer).  Prints ONE JSON line (rank 0).  Under
torchrun every rank runs the same workload on its own GPU with no data-path
collective (independent replicas, weak scaling); `value` is the tokens of
all ranks divided by the slowest rank's time.

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
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral_decode", choices=sorted(I.WORKLOADS))
    ap.add_argument("--shape", default=None,
                    help="T,H,F,E,k: a uniform-routing workload of these sizes instead")
    ap.add_argument("--sweep", action="store_true",
                    help="tokens-per-expert sweep of the workload's shape (own JSON line)")
    ap.add_argument("--train", action="store_true",
                    help="time a training step: moe_forward_train + moe_backward (own JSON line)")
    ap.add_argument("--gated", action="store_true",
                    help="time the layer from hidden states (router projection + routed "
                         "experts + --shared-f shared expert) instead (own JSON line)")
    ap.add_argument("--shared-f", type=int, default=0,
                    help="FFN width of the shared expert for --gated (0 = none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
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
def bench_ours(args, rank, world, local):
    import routing_grouped_expert_gb300 as moe
    import torch.distributed as dist

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[args.workload]
    d = I.make_inputs(wl, dev)
    x, logits, W1, W3, W2 = d["x"], d["logits"], d["W1"], d["W3"], d["W2"]
    ws = moe.Workspace(dev)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    P = wl.T * wl.k

    # routing statistics for the byte accounting (not timed)
    idx, _ = moe.moe_route_topk(logits, wl.k, ws=ws)
    counts = moe.moe_permute(idx, wl.E, ws=ws)[0].cpu()
    touched = int((counts > 0).sum())
    max_count = int(counts.max())

    weight_bytes = acc.expert_weight_bytes(wl.H, wl.F, touched)
    flush = weight_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    nst = moe.FORWARD_STAGES
    for _ in range(args.warmup):
        moe.moe_forward(x, logits, W1, W3, W2, wl.k, out=out, ws=ws)
    st = moe.moe_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {moe.moe_status_string(st)}")

    # Timed region 1 (the value): K plain moe_forward steps.  With the L2 flush
    # between steps, each step is bracketed by its own pair of events so the
    # flush is not counted.
    K = args.steps
    step_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    barrier()
    if clocks:
        time.sleep(0.3)
        clocks.mark_begin()
    t_start.record()
    for i in range(K):
        if flush:
            flush_buf.zero_()
            step_evs[i][0].record()
        moe.moe_forward(x, logits, W1, W3, W2, wl.k, out=out, ws=ws)
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
    ms_per_step = region_ms / K
    value = throughput(world, wl.T, K, region_ms)

    # Timed region 2 (the per-kernel breakdown): K steps of moe_forward_events,
    # one event between consecutive kernels on the launch stream.  The events
    # themselves cost a few microseconds per step, which is why the value
    # above comes from the region without them.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(K)]
    barrier()
    for i in range(K):
        if flush:
            flush_buf.zero_()
        moe.moe_forward_events(x, logits, W1, W3, W2, wl.k, evs[i], out=out, ws=ws)
    barrier()
    stage_ms = [[evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)] for j in range(nst)]
    events_ms_per_step = statistics.fmean(evs[i][0].elapsed_time(evs[i][nst]) for i in range(K))

    # end to end: host activations in, host result out, through the C ABI
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        lh = logits.cpu().pin_memory()
        oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        for _ in range(max(3, args.warmup // 2)):
            moe.moe_forward_host(xh, lh, W1, W3, W2, wl.k, out_host=oh, ws=ws)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            if flush:
                flush_buf.zero_()
            moe.moe_forward_host(xh, lh, W1, W3, W2, wl.k, out_host=oh, ws=ws)
        e1.record()
        barrier()
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
    names = [moe.moe_forward_stage_name(j) for j in range(nst)]
    mean_ms = {n: statistics.fmean(v) for n, v in zip(names, stage_ms)}
    kern_sum = sum(mean_ms.values())
    kernels = {n: {"ms": round(mean_ms[n], 5), "share": round(mean_ms[n] / kern_sum, 4)}
               for n in names}
    # roofline of the dominant kernel
    top = max(mean_ms, key=mean_ms.get)
    kbytes = {"route": acc.route_bytes(wl.T, wl.E, wl.k),
              "scan": 0, "scatter": 4 * P * 4,
              "gather": acc.gather_bytes(wl.T, wl.k, wl.H),
              "fc1": acc.fc1_bytes(wl.H, wl.F, touched, P),
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

    flops = acc.ffn_flops(wl.T, wl.H, wl.F, wl.k)
    lbytes = acc.layer_bytes(wl.T, wl.H, wl.F, wl.E, wl.k, touched)
    t_roof, bound = acc.roofline_seconds(flops, lbytes, peaks["bf16_tflops"] * 1e12,
                                         peaks["hbm_gbs"] * 1e9)
    layer = {"flops": flops, "bytes": lbytes, "t_roof_ms": round(t_roof * 1e3, 4),
             "bound": bound, "frac": round(t_roof / (ms_per_step / 1e3), 4),
             "tflops": round(flops / (ms_per_step / 1e3) / 1e12, 2),
             "hbm_gbs": round(lbytes / (ms_per_step / 1e3) / 1e9, 1)}

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
        "roofline": roof,
        "layer_roofline": layer,
        "kernels": kernels,
        "kernels_timing": ("per-stage CUDA events on the launch stream, in a second timed "
                           f"region of {K} moe_forward_events steps "
                           f"({events_ms_per_step:.4f} ms per step with the events)"),
        "gpu_launches": nst * K,
        "clocks": clocks.summary() if clocks else None,
    }
    if e2e:
        result["e2e"] = e2e
    return result, d, counts


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


def oracle_sampler(wl, d, mem_cap=24 * 2**30, max_pool=64):
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
        step = statistics.median(evs[i][0].elapsed_time(evs[i][nst]) for i in range(K))
        ffn = statistics.median(evs[i][4].elapsed_time(evs[i][6]) for i in range(K))
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
    if args.impl == "reference":
        res = bench_reference(args, rank, world, local)
        if res is not None:
            print(json.dumps(res), flush=True)
    else:
        out = bench_ours(args, rank, world, local)
        if out is not None:
            res, d, _ = out
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
