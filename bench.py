#!/usr/bin/env python
"""Benchmark of one quantized MoE layer's decode step on GB300.

Workload (default): a 128-expert, top-8 MoE layer with D=2048, Dff=768 and
affine 4-bit group-64 experts (the Qwen3-30B-A3B layer shape), decoding one
token per step. x is bf16 N(0,1), the router is bf16 N(0,0.02) with top-k
logit margins >= 1e-2, and expert weights are N(0,0.02) before quantisation.
All data is synthetic and seeded.

A step is one moe_decode_forward call: the router, grouping, gate/up, down
and combine for one cohort. Steps cycle through R resident layer replicas and
P pre-drawn cohorts, so an expert plane read in one step was last read at
least R-1 steps (hundreds of MB of other traffic) earlier and is not
L2-resident.

Output: one JSON line (rank 0). `value` is tokens/s of the whole job over the
timed K steps, which run as a captured CUDA graph; `e2e` is the same metric
through the host-buffer entry point, with the H2D and D2H copies inside the
timed region; `roofline` relates the unique expert bytes per step to the
measured HBM peak.

`--stack L --sweep 1,2,...` instead times a stack of L distinct layers (one
forward per layer per step, e.g. 48 layers and 16 GB of planes) and prints one
line per cohort size of the sweep.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s; unique-expert-byte HBM GB/s vs GB300 peak"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--shape", default="qwen3", choices=["qwen3", "e256", "tiny"])
    ap.add_argument("--n-tokens", type=int, default=1)
    ap.add_argument("--kind", default="independent", choices=["independent", "shared", "disjoint"])
    ap.add_argument("--replicas", type=int, default=16)
    ap.add_argument("--cohorts", type=int, default=64)
    ap.add_argument("--flags", type=int, default=0, help="MOE_FLAG_* for the plan")
    ap.add_argument("--mma-min-tokens", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--stack", type=int, default=0,
                    help="time a stack of this many distinct layers (one step = one forward "
                         "per layer) and print one line per --sweep cohort size")
    ap.add_argument("--sweep", default="1,2,4,8,16,32,64",
                    help="cohort sizes of the --stack run")
    ap.add_argument("--no-chain", action="store_true",
                    help="--stack: one moe_decode_forward call per layer instead of one "
                         "moe_decode_forward_layers chain per step")
    ap.add_argument("--phases", action="store_true",
                    help="also time the fused kernel's phases (router / gate-up / down)")
    ap.add_argument("--sustain-seconds", type=float, default=1.5,
                    help="graph replays before the timed ones, while clocks are sampled")
    ap.add_argument("--runs", type=int, default=7,
                    help="timed replays of the K-step graph (value = the median run)")
    return ap.parse_args()


SEEDS = {"qwen3": 1, "e256": 3, "tiny": 0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# single-launch kernel, from an ncu capture of the same workload (one layer,
# cold caches), keyed by (shape, n_tokens), with the unique experts of the
# captured cohort and a hash of the kernel sources it was built from. The
# number is reported only while the sources still hash the same, scaled to the
# timed steps' mean unique-expert count (traffic grows with it).
KERNEL_SOURCES = ("decode_step.cu", "ptx.cuh", "routing.cuh", "moe_internal.h")
TRAFFIC = {
    ("qwen3", 1): {"bytes": 21859328 + 0, "unique": 8, "src": "941f32f5a6607795"},
    ("qwen3", 8): {"bytes": 138673920 + 2810624, "unique": 52, "src": "941f32f5a6607795"},
}


def kernel_src_hash():
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "quantized_moe_decode_softmax_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch(shape_name, n, avg_unique):
    t = TRAFFIC.get((shape_name, n))
    if t is None or t["src"] != kernel_src_hash():
        return None
    return t["bytes"] * avg_unique / t["unique"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_tensor_peak():
    """bf16 dense TFLOP/s: the sustained figure (a kernel timed inside a long
    step), else the burst one, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        if "bf16_tflops_sustained" in p:
            return float(p["bf16_tflops_sustained"]), "measured sustained"
        return float(p["bf16_tflops"]), "measured burst"
    return 1700.0, "fallback sustained"


def step_flops(shape, n):
    """Algorithmic flops of one step: the router GEMV and, per (token, slot),
    the gate, up and down products (6 D Dff multiply-adds counted as 2 flops)."""
    return 2.0 * n * shape.E * shape.D + n * shape.top_k * 6.0 * shape.D * shape.F


# ----------------------------------------------------------------------------
# clocks sampler
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smmax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smmax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smmax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# distributed helpers (one process per GPU; independent replicas)
# ----------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device])
        else:
            pg.barrier()


def max_over_ranks(pg, value: float, device=None) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# oracle (CPU) timing: the reference arm and the cpu_baseline key
# ----------------------------------------------------------------------------
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_sample(shape_name, n, kind, cohorts, seconds, threads=None):
    """Time the CPU oracle on cohorts of the workload for about `seconds`, on
    `threads` OpenMP threads (default: every host core)."""
    import numpy as np

    import moe_synth as ms
    import oracle
    shape = ms.SHAPES[shape_name]
    seed = SEEDS[shape_name]
    router_w, bias = ms.draw_router(shape, seed, 0)
    xs = [ms.draw_tokens(shape, router_w, bias, seed, 0, n, kind, cohort=c) for c in range(cohorts)]
    experts = sorted({e for x in xs for e in ms.routed_experts(x, router_w, bias, shape.top_k)})
    lay = ms.make_layer(shape, seed, 0, experts)
    threads = oracle.set_threads(threads or os.cpu_count() or 1)
    oracle.moe_forward(xs[0], router_w, bias, lay.planes, shape.top_k)  # warm
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle.moe_forward(xs[steps % cohorts], router_w, bias, lay.planes, shape.top_k)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": n * steps / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{steps} steps of n_tokens={n} ({kind} cohorts), {el:.1f} s, "
                      f"OpenMP over (token, expert) slots"}, steps, el


def cpu_baseline(args):
    """The oracle on all host cores, plus its single-thread leg."""
    seconds = max(1.0, min(30.0, args.cpu_seconds))
    cohorts = min(args.cohorts, 16)
    cb, _, _ = oracle_sample(args.shape, args.n_tokens, args.kind, cohorts, seconds)
    one, _, _ = oracle_sample(args.shape, args.n_tokens, args.kind, cohorts, seconds, threads=1)
    cb["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": one["cores"],
                           "sample": one["sample"]}
    return cb


def run_reference(args, world, rank, pg):
    """The oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    shape_name, n = args.shape, args.n_tokens
    seconds = max(1.0, min(30.0, args.cpu_seconds))
    cb, steps, el = oracle_sample(shape_name, n, args.kind, min(args.cohorts, 16), seconds)
    one, _, _ = oracle_sample(shape_name, n, args.kind, min(args.cohorts, 16), min(seconds, 5.0),
                              threads=1)
    cb["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": one["cores"],
                           "sample": one["sample"]}
    line = {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": 1, "ms_per_step": 1000.0 * el / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(args),
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(args):
    import moe_synth as ms
    shape = ms.SHAPES[args.shape]
    names = {"qwen3": "qwen3-30b-a3b-shaped MoE layer", "e256": "256-expert top-6 MoE layer",
             "tiny": "tiny MoE layer"}
    return {"workload": f"{names[args.shape]} decode, n_tokens={args.n_tokens}",
            "E": shape.E, "top_k": shape.top_k, "D": shape.D, "Dff": shape.F,
            "quant": "affine 4-bit, group 64, bf16 scale+bias", "n_tokens": args.n_tokens,
            "cohorts": args.kind, "global_batch": args.n_tokens * args.gpus,
            "l2": f"{args.replicas} resident layer replicas cycled, {args.cohorts} cohorts",
            "parallelism": f"replicas x{args.gpus}"}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, world, rank, local, pg):
    import numpy as np
    import torch

    import moe_synth as ms
    import quantized_moe_decode_softmax_gb300 as q

    shape = ms.SHAPES[args.shape]
    seed = SEEDS[args.shape]
    n = args.n_tokens
    workers = max(1, min(16, os.cpu_count() or 1))

    # host-side generation (spawn pool: safe before or after CUDA init)
    lay = ms.make_layer(shape, seed, 0, workers=workers)
    cohorts = [ms.draw_tokens(shape, lay.router_w, lay.router_bias, seed, 0, n, args.kind, cohort=c)
               for c in range(args.cohorts)]
    U_of = [len(ms.routed_experts(x, lay.router_w, lay.router_bias, shape.top_k)) for x in cohorts]

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    base = q.DeviceLayer.from_host(ms.router_storage(shape, lay.router_w), lay.router_bias,
                                   lay.planes, shape.top_k, device=dev)
    reps = [base]
    for _ in range(args.replicas - 1):
        planes = {f: t.clone() for f, t in base.planes.items()}
        rb = None if base.router_bias is None else base.router_bias.clone()
        reps.append(q.DeviceLayer(base.router_w.clone(), rb, planes, base.E, base.top_k, base.D,
                                  base.Dff))
    del lay
    act = torch.bfloat16 if shape.act_dtype == "bf16" else torch.float32

    def to_dev(x):
        st = ms.x_storage(shape, x)
        t = torch.from_numpy(st.view(np.int16) if st.dtype == np.uint16 else st)
        return t.to(dev).view(act) if st.dtype == np.uint16 else t.to(dev)

    xs = [to_dev(x) for x in cohorts]
    outs = [torch.empty((n, shape.D), dtype=act, device=dev) for _ in range(2)]
    layer = q.MoeDecodeLayer(shape.E, shape.top_k, shape.D, shape.F, max_tokens=max(n, 1),
                             act_dtype=shape.act_dtype, flags=args.flags,
                             mma_min_tokens=args.mma_min_tokens)
    stream = torch.cuda.Stream(device=dev)
    K, W = args.steps, args.warmup

    def step(i, s):
        layer.forward(xs[i % len(xs)], reps[i % len(reps)], outs[i % 2], stream=s)

    c0 = q.moe_plan_launch_count(layer.plan)
    with torch.cuda.stream(stream):
        for i in range(W):
            step(i, stream)
    stream.synchronize()
    layer.check()
    launches_per_step = (q.moe_plan_launch_count(layer.plan) - c0) / max(W, 1)

    # capture exactly K steps; a second graph brackets each step with events
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            step(W + i, stream)
    ev_graph = None
    try:
        ev = [(torch.cuda.Event(enable_timing=True, external=True),
               torch.cuda.Event(enable_timing=True, external=True)) for _ in range(K)]
        ev_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ev_graph, stream=stream):
            for i in range(K):
                ev[i][0].record(stream)
                step(W + i, stream)
                ev[i][1].record(stream)
    except TypeError:
        ev_graph = None

    # sustained replays for the clock record, then the timed replay
    sampler = None if args.no_clocks else ClockSampler(local)
    with torch.cuda.stream(stream):
        graph.replay()
        stream.synchronize()
        if sampler:
            sampler.start()
        t_end = time.perf_counter() + args.sustain_seconds
        while time.perf_counter() < t_end:
            graph.replay()
            stream.synchronize()
        # R timed replays of the K-step graph, each bracketed by a barrier and a
        # synchronize; the line reports the median run and the range
        run_ms = []
        for _ in range(max(1, args.runs)):
            barrier(pg, local)
            torch.cuda.synchronize()
            start = torch.cuda.Event(enable_timing=True)
            stop = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            graph.replay()
            stop.record(stream)
            stop.synchronize()
            torch.cuda.synchronize()
            barrier(pg, local)
            run_ms.append(max_over_ranks(pg, start.elapsed_time(stop), dev))
        clocks = sampler.stop() if sampler else None
    layer.check()
    elapsed_ms = statistics.median(run_ms)
    ms_per_step = elapsed_ms / K

    # per-step device time (each step's events), same inputs
    kernel_ms = None
    if ev_graph is not None:
        with torch.cuda.stream(stream):
            ev_graph.replay()
            stream.synchronize()
        kernel_ms = sum(a.elapsed_time(b) for a, b in ev) / K

    # e2e: host buffers through the public API, copies inside the timed region
    E2E = max(1, min(args.e2e_steps, K))
    x_host = [xs[i % len(xs)].cpu().pin_memory() for i in range(min(E2E, len(xs)))]
    out_host = torch.empty((n, shape.D), dtype=act).pin_memory()
    with torch.cuda.stream(stream):
        layer.forward_host(x_host[0], reps[0], out_host, stream=stream)
        barrier(pg, local)
        t0 = time.perf_counter()
        for i in range(E2E):
            layer.forward_host(x_host[i % len(x_host)], reps[i % len(reps)], out_host, stream=stream)
        t1 = time.perf_counter()
    e2e_s = max_over_ranks(pg, t1 - t0, dev)
    esize = 2 if shape.act_dtype == "bf16" else 4

    # algorithmic bytes of the timed steps
    steps_U = [U_of[(W + i) % len(U_of)] for i in range(K)]
    avg_U = sum(steps_U) / K
    act_bytes = n * shape.D * esize * 2
    bytes_per_step = avg_U * shape.plane_bytes + act_bytes
    router_bytes = shape.E * shape.D * esize
    peak, peak_kind = load_peaks()
    # the dominant kernel's average launch duration: the K-step graph replay
    # timed with events on the launching stream, divided by its launches (one
    # per step on the single-launch path)
    t_kernel = ms_per_step / max(launches_per_step, 1.0) / 1000.0
    achieved = bytes_per_step / max(launches_per_step, 1.0) / t_kernel / 1e9
    value = world * n * K / (elapsed_ms / 1000.0)

    phases = None
    if args.phases:
        phases = phase_split(q, shape, args, xs, reps, dev, n)

    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": None if launches_per_step != 1.0
                else traffic_per_launch(args.shape, n, avg_U),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback",
                "kernel_us": t_kernel * 1e6,
                "timing": "CUDA events around the K-step graph replay on the "
                          "launching stream / launches",
                "kernel_us_event_bracketed": None if kernel_ms is None
                else kernel_ms * 1000.0}
    if n > 64:
        # prefill cohorts: a grouped GEMM per expert, bound by the tensor cores
        tpeak, tkind = load_tensor_peak()
        tflops = step_flops(shape, n) / (ms_per_step / 1000.0) / 1e12
        roofline = {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": tflops / tpeak, "traffic": None,
                    "peak_source": f"{tkind} (MEASURED_PEAKS.json bf16 dense)",
                    "flops_per_step": step_flops(shape, n),
                    "timing": "whole step (router, routing, grouped GEMMs, combine) over the "
                              "K-step graph replay; tcgen05 grouped GEMMs",
                    "hbm_frac_unique_expert_bytes": achieved * launches_per_step / peak}
    if rank == 0:
        cb = None if args.no_cpu_baseline else cpu_baseline(args)
        tok = sorted(world * n * K / (m / 1000.0) for m in run_ms)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True,
            "runs": {"n": len(run_ms), "value_is": "median run",
                     "ms_per_step": {"min": min(run_ms) / K, "median": ms_per_step,
                                     "max": max(run_ms) / K},
                     "tokens_per_s": {"min": tok[0], "median": value, "max": tok[-1]}},
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; random-init weights of the layer shape)",
            "config": workload_config(args),
            "hbm_gbs_unique_expert_bytes": bytes_per_step / (ms_per_step / 1000.0) / 1e9,
            "unique_experts_per_step": avg_U,
            "bytes_per_step": bytes_per_step,
            "router_bytes_per_step": router_bytes,
            "roofline": roofline,
            "e2e": {"value": world * n * E2E / e2e_s, "unit": "tokens/s",
                    "h2d_bytes_per_step": n * shape.D * esize,
                    "d2h_bytes_per_step": n * shape.D * esize, "steps": E2E},
            "gpu_launches": int(round(K * launches_per_step)),
            "clocks": clocks,
            "cpu_baseline": cb,
        }
        if phases is not None:
            line["phases_us"] = phases
        print(json.dumps(line), flush=True)
    layer.close()


def phase_split(q, shape, args, xs, reps, dev, n, steps=50):
    """Median over steps of the fused kernel's phase durations (us), each phase
    taken as the latest CTA's timestamp minus the earliest start."""
    import numpy as np
    import torch
    lay = q.MoeDecodeLayer(shape.E, shape.top_k, shape.D, shape.F, max_tokens=max(n, 1),
                           act_dtype=shape.act_dtype, flags=q.MOE_FLAG_PHASE_TIMES)
    out = torch.empty((n, shape.D), dtype=xs[0].dtype, device=dev)
    per, cnt = [], []
    for i in range(steps):
        lay.forward(xs[i % len(xs)], reps[(i * 7) % len(reps)], out)
        t = q.moe_get_phase_times(lay.plan)
        t0 = t[:, 0].min()
        per.append((t[:, :8] - t0).max(axis=0) / 1000.0)
        cnt.append(np.concatenate([t[:, 8:13].mean(axis=0) / 1000.0, t[:, 13:15].mean(axis=0)]))
    lay.close()
    med = np.median(np.array(per), axis=0)
    cm = np.median(np.array(cnt), axis=0)
    names = q.PHASES
    res = {f"{names[i]}_end": round(float(med[i]), 3) for i in range(1, 8)}
    for j, nm in enumerate(names[8:15]):
        res[nm] = round(float(cm[j]), 3)
    return res


# ----------------------------------------------------------------------------
# layer stack: L distinct layers, one forward per layer per step
# ----------------------------------------------------------------------------
def run_stack(args, world, rank, local, pg):
    """A stack of `args.stack` layers of one shape, each with its own seeded
    weights and router (about 14.5 GB of expert planes for 48 Qwen3-shaped
    layers). A step runs one forward per layer, in layer order, each on a cohort
    drawn for that layer's router (so routing keeps its per-layer diversity; no
    attention or residual kernels run between layers). One JSON line per cohort
    size of --sweep: tokens/s through the whole stack, the per-layer time, and
    the unique-expert bytes against the HBM peak."""
    import numpy as np
    import torch

    import moe_synth as ms
    import quantized_moe_decode_softmax_gb300 as q

    shape = ms.SHAPES[args.shape]
    seed = SEEDS[args.shape]
    L = args.stack
    sizes = [int(v) for v in args.sweep.split(",") if v.strip()]
    workers = max(1, min(16, os.cpu_count() or 1))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    act = torch.bfloat16 if shape.act_dtype == "bf16" else torch.float32
    t_gen = time.perf_counter()
    layers, routers = [], []
    for l in range(L):
        lay = ms.make_layer(shape, seed, l, workers=workers)
        layers.append(q.DeviceLayer.from_host(ms.router_storage(shape, lay.router_w), lay.router_bias,
                                              lay.planes, shape.top_k, device=dev))
        routers.append((lay.router_w, lay.router_bias))
        del lay
    t_gen = time.perf_counter() - t_gen
    P = 4  # cohorts per layer, cycled over the steps
    peak, peak_kind = load_peaks()
    esize = 2 if shape.act_dtype == "bf16" else 4

    def to_dev(x):
        st = ms.x_storage(shape, x)
        t = torch.from_numpy(st.view(np.int16) if st.dtype == np.uint16 else st)
        return t.to(dev).view(act) if st.dtype == np.uint16 else t.to(dev)

    for n in sizes:
        xs, U_of = [], []
        for l in range(L):
            rw, rb = routers[l]
            cs = [ms.draw_tokens(shape, rw, rb, seed, l, n, args.kind, cohort=c) for c in range(P)]
            xs.append([to_dev(x) for x in cs])
            U_of.append([len(ms.routed_experts(x, rw, rb, shape.top_k)) for x in cs])
        outs = [torch.empty((n, shape.D), dtype=act, device=dev) for _ in range(2)]
        layer = q.MoeDecodeLayer(shape.E, shape.top_k, shape.D, shape.F, max_tokens=n,
                                 act_dtype=shape.act_dtype, flags=args.flags,
                                 mma_min_tokens=args.mma_min_tokens)
        stream = torch.cuda.Stream(device=dev)
        # a step is L forwards: at most 20 steps per graph (the graph holds K * L
        # forwards), at least 3 warm-up steps
        K, W = max(1, min(args.steps, 20)), max(3, min(args.warmup, 5))

        def step(i):
            if args.no_chain:
                for l in range(L):
                    layer.forward(xs[l][i % P], layers[l], outs[l % 2], stream=stream)
            else:
                layer.forward_layers([(xs[l][i % P], layers[l], outs[l % 2]) for l in range(L)],
                                     stream=stream)

        c0 = q.moe_plan_launch_count(layer.plan)
        with torch.cuda.stream(stream):
            for i in range(W):
                step(i)
        stream.synchronize()
        layer.check()
        launches_per_step = (q.moe_plan_launch_count(layer.plan) - c0) / max(W, 1)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(K):
                step(W + i)
        sampler = None if args.no_clocks else ClockSampler(local)
        with torch.cuda.stream(stream):
            graph.replay()
            stream.synchronize()
            if sampler:
                sampler.start()
            t_end = time.perf_counter() + args.sustain_seconds
            while time.perf_counter() < t_end:
                graph.replay()
                stream.synchronize()
            barrier(pg, local)
            torch.cuda.synchronize()
            start = torch.cuda.Event(enable_timing=True)
            stop = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            graph.replay()
            stop.record(stream)
            stop.synchronize()
            torch.cuda.synchronize()
            barrier(pg, local)
            clocks = sampler.stop() if sampler else None
        layer.check()
        elapsed_ms = max_over_ranks(pg, start.elapsed_time(stop), dev)
        ms_per_step = elapsed_ms / K
        # phase split of one layer's single-launch step (fused cohorts only)
        phases = (phase_split(q, shape, args, xs[0], [layers[0]], dev, n)
                  if args.phases and n <= 8 else None)
        avg_U = sum(U_of[l][(W + i) % P] for i in range(K) for l in range(L)) / K
        bytes_per_step = avg_U * shape.plane_bytes + L * n * shape.D * esize * 2
        achieved = bytes_per_step / (ms_per_step / 1000.0) / 1e9
        if rank == 0:
            line = {
                "metric": METRIC, "value": world * n * K / (elapsed_ms / 1000.0), "unit": "tokens/s",
                "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded; random-init weights of the layer shape)",
                "config": {"workload": f"{L}-layer stack of {shape.E}-expert top-{shape.top_k} "
                                       f"D={shape.D} Dff={shape.F} MoE layers, n_tokens={n}",
                           "layers": L, "n_tokens": n, "cohorts": args.kind,
                           "calls": "one forward call per layer" if args.no_chain
                           else "one moe_decode_forward_layers chain per step",
                           "expert_plane_bytes": L * shape.E * shape.plane_bytes,
                           "l2": "every layer's planes are read once per step (stack >> L2)",
                           "parallelism": f"replicas x{world}"},
                "per_layer_us": ms_per_step * 1000.0 / L,
                "layer_tokens_per_s": world * n * K * L / (elapsed_ms / 1000.0),
                "unique_experts_per_layer": avg_U / L,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "traffic": None,
                             "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                             if peak_kind == "measured" else "fallback",
                             "timing": "CUDA events around the K-step graph replay"},
                "gpu_launches": int(round(K * launches_per_step)),
                "launches_per_layer": launches_per_step / L,
                "clocks": clocks,
                "phases_us": phases,
                "stack_build_s": t_gen,
            }
            print(json.dumps(line), flush=True)
        layer.close()
        del xs, outs, graph


def main():
    args = parse_args()
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank, pg)
    elif args.stack > 0:
        run_stack(args, world, rank, local, pg)
    else:
        run_ours(args, world, rank, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
