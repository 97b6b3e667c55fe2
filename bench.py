#!/usr/bin/env python3
"""Bench: MXFP4 weight-streaming decode/verify step on GB300.

One step = one weight-streaming call over one batch of decode tokens
(headline workload: T=4 verify step, K=N=7168 dense projection). Prints one
JSON line (rank 0). Metric: effective HBM GB/s, where bytes = 0.53125*N*K
(packed weights + scales actually read) + 2*T*K (x) + 2*T*N (y).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-workloads]

Timing: the timed steps are CUDA-graph replays of back-to-back calls that
cycle through enough independent weight copies to exceed 2x L2, so every
call streams its weights from HBM. CUDA events on the launching stream
bracket the whole region (device time); each call is one kernel launch, so
the average launch duration behind the roofline is the region time over
the calls (back to back, the gaps between launches included). Events
between graph replays give the per-replay spread (p10/p50/p90 of the
per-call time). Clocks are sampled with nvidia-smi while each workload runs.

Besides the headline line's `value`, the default run times every other
configuration of the method (the T=1 K=N=1024 linear, the LM head, the FFN
token sweep, the fused FFN chain and the grouped MoE at T=32 and T=128)
under a `workloads` key, each with its own clock summary.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s (% of GB300 peak) and us/call, MXFP4 GEMM at T=1-32"
FALLBACK_HBM_GBS = 6800.0  # fallback peak when no measured peak file is present
KERNEL_SOURCES = ["mxfp4_weight_streaming_gb300/csrc/linear.cu", "mxfp4_weight_streaming_gb300/csrc/engine.cuh",
                  "mxfp4_weight_streaming_gb300/csrc/engine_layout.h",
                  "mxfp4_weight_streaming_gb300/csrc/device_common.cuh",
                  "mxfp4_weight_streaming_gb300/csrc/f4_linear.cu", "mxfp4_weight_streaming_gb300/csrc/tc_common.cuh"]

WORKLOADS = {
    "linear_t1_k1024_n1024": dict(t=1, k=1024, n=1024, seed=0, x64=False),
    "verify_t4_k7168_n7168": dict(t=4, k=7168, n=7168, seed=1, x64=False),
    "lmhead_t4_k7168_n129280": dict(t=4, k=7168, n=129280, seed=2, x64=True),
    "ffn_up_t1_k7168_n18432": dict(t=1, k=7168, n=18432, seed=3, x64=False),
    "ffn_up_t2_k7168_n18432": dict(t=2, k=7168, n=18432, seed=3, x64=False),
    "ffn_up_t4_k7168_n18432": dict(t=4, k=7168, n=18432, seed=3, x64=False),
    "ffn_up_t8_k7168_n18432": dict(t=8, k=7168, n=18432, seed=3, x64=False),
    "ffn_up_t16_k7168_n18432": dict(t=16, k=7168, n=18432, seed=3, x64=False),
    "ffn_up_t32_k7168_n18432": dict(t=32, k=7168, n=18432, seed=3, x64=False),
}
DEFAULT_WORKLOAD = "verify_t4_k7168_n7168"
MOE_WORKLOAD = "moe_e256_top8_t32"
MOE = dict(t=32, e=256, top_k=8, hidden=7168, inter=2048, seed=4)
# The grouped MoE at a larger token count (every expert receives several
# chunks of tokens), timed beside the T=32 configuration.
MOE_LARGE_T = 128
# Fused dense FFN chain (mxfp4_ffn): W1 [2*inter, hidden] then W2 [hidden,
# inter], hidden 7168 and inter 9216 (the FFN width of the up projection).
FFN_CHAIN = {f"ffn_chain_t{t}_h7168_i9216": dict(t=t, hidden=7168, inter=9216, seed=3) for t in (1, 2, 4)}


def algorithmic_bytes(t: int, k: int, n: int) -> int:
    return n * k // 2 + n * k // 32 + 2 * t * k + 2 * t * n


def reduce_max(x: float, device) -> float:
    """Maximum of x over the ranks of the job (x itself without a process
    group): every rank waits for the slowest one."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    if torch.distributed.get_world_size() == 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_call: int, calls_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return bytes_per_call * calls_per_rank * world / seconds / 1e9


def kernel_digest() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def hbm_peak():
    """(GB/s, source) from the measured-peaks file, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBps", "hbm_gb_s", "copy_gbs"):
                if key in d:
                    return float(d[key]), "measured"
            for v in d.values():
                if isinstance(v, dict):
                    for key in ("hbm_gbs", "hbm_GBps"):
                        if key in v:
                            return float(v[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        ent = d.get(workload)
        if ent and ent.get("kernel_digest") == kernel_digest():
            return int(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [p for (ts, p) in self.samples if t0 <= ts <= t1] or [p for (_, p) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_median": statistics.median(power) if power else None}


# ---------------------------------------------------------------- our arm
PLAN_KERNELS = {
    0: "mxfp4::stream_kernel<DenseProblem, whole K> (mma.sync)",
    1: "mxfp4::stream_kernel<DenseProblem, K in parts> (mma.sync)",
    2: "mxfp4::stream_kernel<DenseProblem, cluster split of K> (mma.sync)",
    3: "mxfp4::tc::tc_linear_kernel (tcgen05.mma kind::mxf8f6f4 block-scaled)",
    4: "mxfp4::f4::f4_linear_kernel (tcgen05.mma kind::mxf4 block-scaled, packed E2M1 weights and digit pieces)",
}


def dense_kernel_name(t: int, k: int, n: int) -> str:
    import mxfp4_weight_streaming_gb300 as mx
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    smem = getattr(props, "shared_memory_per_block_optin", 232448)
    plan = mx.linear_plan(t, k, n, props.multi_processor_count, smem)
    return PLAN_KERNELS.get(plan["mode"], f"mode {plan['mode']}") + f" [{plan['ctas']} CTAs, cluster {plan['cluster']}]"


def setup_dense(wl: dict, device, cache=None):
    import torch

    import mxfp4_weight_streaming_gb300 as mx
    import synth

    t, k, n = wl["t"], wl["k"], wl["n"]
    key = (wl["seed"], k, n, wl["x64"])
    if cache is not None and key in cache:
        wq, ws = cache[key]
    else:
        w = synth.weights(wl["seed"], n, k, device=device, x64_blocks=wl["x64"])
        wq, ws = mx.quantize(w)
        del w
        if cache is not None:
            cache.clear()
            cache[key] = (wq, ws)
    x = synth.tokens(wl["seed"], t, k, device=device)
    y = torch.empty((t, n), dtype=torch.bfloat16, device=device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    wbytes = wq.numel() + ws.numel()
    copies = max(1, math.ceil(2 * l2 / wbytes) + 1) if wbytes < 2 * l2 else 1
    wqs = [wq] + [wq.clone() for _ in range(copies - 1)]
    wss = [ws] + [ws.clone() for _ in range(copies - 1)]
    torch.cuda.synchronize()
    return dict(x=x, y=y, wqs=wqs, wss=wss, copies=copies, t=t, k=k, n=n, l2=l2)


def percentiles(per_call_us):
    xs = sorted(per_call_us)

    def q(f):
        return xs[min(len(xs) - 1, max(0, int(round(f * (len(xs) - 1)))))]

    return {"p10": round(q(0.1), 3), "p50": round(q(0.5), 3), "p90": round(q(0.9), 3), "max": round(xs[-1], 3),
            "replays": len(xs)}


class GraphTimer:
    """G back-to-back calls captured once; timed by events around the whole
    region (the headline) and between replays (the spread)."""

    def __init__(self, call, G, stream):
        import torch
        self.G = G
        self.stream = stream
        with torch.cuda.stream(stream):
            for i in range(3):
                call(i)  # first calls set per-device state before capture
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            for i in range(G):
                call(i)

    def soak(self, seconds):
        import torch
        end = time.time() + seconds
        with torch.cuda.stream(self.stream):
            while time.time() < end:
                self.graph.replay()
                self.stream.synchronize()
        torch.cuda.synchronize()

    def run(self, replays):
        """(total ms, per-replay per-call us list)."""
        import torch
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
        with torch.cuda.stream(self.stream):
            evs[0].record(self.stream)
            for r in range(replays):
                self.graph.replay()
                evs[r + 1].record(self.stream)
        evs[-1].synchronize()
        per = [evs[r].elapsed_time(evs[r + 1]) * 1e3 / self.G for r in range(replays)]
        return evs[0].elapsed_time(evs[-1]), per


def gpu_index():
    import torch
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    return torch.cuda.current_device() if vis is None else int(vis.split(",")[0])


def run_ours(args, wl_name: str, rank: int, world: int, device, with_cpu_baseline: bool, clocks):
    import torch

    import mxfp4_weight_streaming_gb300 as mx

    wl = WORKLOADS[wl_name]
    st = setup_dense(wl, device)
    t, k, n = st["t"], st["k"], st["n"]
    stream = torch.cuda.Stream(device)
    sp = stream.cuda_stream
    lib = mx.load()
    xp, yp = st["x"].data_ptr(), st["y"].data_ptr()
    wq_ptrs = [a.data_ptr() for a in st["wqs"]]
    ws_ptrs = [a.data_ptr() for a in st["wss"]]

    def call(i):
        rc = lib.mxfp4_linear(xp, t, k, wq_ptrs[i % st["copies"]], ws_ptrs[i % st["copies"]], n, yp, sp)
        if rc != 0:
            raise RuntimeError(mx.strerror(rc))

    # Graph of G back-to-back calls (a multiple of the weight-copy count);
    # the timed region is a whole number of replays.
    G = max(st["copies"], min(args.steps, 256 // st["copies"] * st["copies"] or st["copies"]))
    G = min(G, max(1, args.steps))
    replays = max(1, args.steps // G)
    steps = replays * G
    timer = GraphTimer(call, G, stream)
    timer.soak(1.0)  # keep the GPU on this workload so clock samples mean something
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
    stream.synchronize()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    elapsed_ms, per_call = timer.run(replays)
    wall1 = time.time()
    torch.cuda.synchronize()
    if world > 1:
        elapsed_ms = reduce_max(elapsed_ms, device)
        torch.distributed.barrier()

    # End to end through the public API: pinned host x in, host y out, every step.
    x_host = st["x"].cpu().pin_memory()
    y_host = torch.empty((t, n), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(1, min(steps, 2000))
    with torch.cuda.stream(stream):
        for i in range(3):
            st["x"].copy_(x_host, non_blocking=True)
            mx.linear(st["x"], st["wqs"][i % st["copies"]], st["wss"][i % st["copies"]], out=st["y"], stream=stream)
            y_host.copy_(st["y"], non_blocking=True)
        stream.synchronize()
        e0 = time.perf_counter()
        for i in range(e2e_steps):
            st["x"].copy_(x_host, non_blocking=True)
            mx.linear(st["x"], st["wqs"][i % st["copies"]], st["wss"][i % st["copies"]], out=st["y"], stream=stream)
            y_host.copy_(st["y"], non_blocking=True)
            stream.synchronize()
        e1 = time.perf_counter()

    bytes_call = algorithmic_bytes(t, k, n)
    us_call = elapsed_ms * 1e3 / steps
    value = job_gbps(bytes_call, steps, world, elapsed_ms * 1e-3)
    peak, peak_src = hbm_peak()
    # Average launch duration over the timed region: one kernel per call,
    # launched back to back, so region time / calls (gaps included).
    avg_launch_ms = elapsed_ms / steps
    achieved = bytes_call / (avg_launch_ms * 1e-3) / 1e9
    e2e_us = reduce_max((e1 - e0) * 1e6 / e2e_steps, device) if world > 1 else (e1 - e0) * 1e6 / e2e_steps
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / steps,
        "us_per_call": round(us_call, 4),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4xbf16->f32",
        "data": "synthetic (seeded counter-based N(0,0.02) weights, N(0,1) bf16 tokens)",
        "config": {"workload": wl_name, "T": t, "K": k, "N": n, "bytes_per_call": bytes_call,
                   "weight_copies": st["copies"], "l2_bytes": st["l2"],
                   "l2_policy": "rotating weight copies (> 2x L2) so every call streams from HBM",
                   "timing": f"{replays} CUDA graph replays of {G} back-to-back calls; device events around the "
                             f"region", "parallelism": f"replicas x{world}"},
        "spread_us_per_call": percentiles(per_call),
        "e2e": {"value": round(job_gbps(bytes_call, 1, world, e2e_us * 1e-6), 2), "unit": "GB/s",
                "us_per_call": round(e2e_us, 3),
                "h2d_bytes_per_step": 2 * t * k, "d2h_bytes_per_step": 2 * t * n},
        "gpu_launches": steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(wl_name),
                     "peak_source": f"{peak_src} (HBM copy bandwidth)",
                     "kernel": dense_kernel_name(t, k, n), "avg_launch_us": round(avg_launch_ms * 1e3, 4),
                     "algorithmic_bytes_per_launch": bytes_call},
        "clocks": clocks.summary(wall0 - 1.5, wall1 + 0.1),
    }
    # Time x median SM clock: SM cycles per call, comparable across runs
    # whose clocks differ.
    if res["clocks"].get("sm_mhz"):
        res["kcycles_per_call"] = round(us_call * res["clocks"]["sm_mhz"] / 1e3, 3)
    if with_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl_name)
    return res


def measure_dense(wl_name: str, device, cache, clocks, calls_target: int = 2000, replays: int = 12):
    """One extra dense workload: per-call time, GB/s, fraction of peak and
    the spread over graph replays, with its own clock samples."""
    import torch

    import mxfp4_weight_streaming_gb300 as mx

    wl = WORKLOADS[wl_name]
    st = setup_dense(wl, device, cache)
    t, k, n = st["t"], st["k"], st["n"]
    stream = torch.cuda.Stream(device)
    sp = stream.cuda_stream
    lib = mx.load()
    xp, yp = st["x"].data_ptr(), st["y"].data_ptr()
    wq_ptrs = [a.data_ptr() for a in st["wqs"]]
    ws_ptrs = [a.data_ptr() for a in st["wss"]]

    def call(i):
        rc = lib.mxfp4_linear(xp, t, k, wq_ptrs[i % st["copies"]], ws_ptrs[i % st["copies"]], n, yp, sp)
        if rc != 0:
            raise RuntimeError(mx.strerror(rc))

    G = max(st["copies"], min(256, calls_target // replays) // st["copies"] * st["copies"])
    timer = GraphTimer(call, G, stream)
    timer.soak(0.4)
    wall0 = time.time()
    ms, per_call = timer.run(replays)
    wall1 = time.time()
    calls = replays * G
    nbytes = algorithmic_bytes(t, k, n)
    us = ms * 1e3 / calls
    peak, _ = hbm_peak()
    gbs = nbytes / (us * 1e-6) / 1e9
    del st
    return {"us_per_call": round(us, 3), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
            "spread_us_per_call": percentiles(per_call), "calls": calls, "bytes_per_call": nbytes,
            "kernel": dense_kernel_name(t, k, n), "launches_per_call": 1,
            "clocks": clocks.summary(wall0 - 0.5, wall1 + 0.1)}


# ------------------------------------------------------------- MoE arm
def moe_expert_bytes(hidden: int, inter: int) -> int:
    return 2 * inter * (hidden // 2 + hidden // 32) + hidden * (inter // 2 + inter // 32)


def ffn_chain_bytes(t: int, hidden: int, inter: int) -> int:
    return int(0.53125 * 3 * inter * hidden) + 2 * t * hidden + 2 * t * hidden


def measure_ffn_chain(wl_name: str, device, clocks, calls_target: int = 1200, replays: int = 12):
    """Dense FFN chain (one mxfp4_ffn call: for t <= 4 with hidden and inter
    multiples of 512, two packed-E2M1 launches chained by programmatic
    dependent launch; otherwise one cooperative launch plus a 4-byte
    memset): per-call time and GB/s of W1 + W2 (+ x, y)."""
    import torch

    import mxfp4_weight_streaming_gb300 as mx
    import synth

    wl = FFN_CHAIN[wl_name]
    t, hidden, inter, seed = wl["t"], wl["hidden"], wl["inter"], wl["seed"]
    w1q, w1s = mx.quantize(synth.weights(seed, 2 * inter, hidden, device=device))
    w2q, w2s = mx.quantize(synth.weights(seed, hidden, inter, tid=synth.TID_W2, device=device))
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    wbytes = w1q.numel() + w1s.numel() + w2q.numel() + w2s.numel()
    copies = max(1, math.ceil(2 * l2 / wbytes) + 1) if wbytes < 2 * l2 else 1
    sets = [(w1q, w1s, w2q, w2s)] + [tuple(a.clone() for a in (w1q, w1s, w2q, w2s)) for _ in range(copies - 1)]
    ptrs = [tuple(a.data_ptr() for a in st) for st in sets]
    x = synth.tokens(seed, t, hidden, device=device)
    y = torch.empty((t, hidden), dtype=torch.bfloat16, device=device)
    ws = torch.empty(mx.mxfp4_ffn_workspace_size(t, hidden, inter), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)
    lib = mx.load()

    def call(i):
        p = ptrs[i % copies]
        rc = lib.mxfp4_ffn(x.data_ptr(), t, hidden, p[0], p[1], p[2], p[3], inter, y.data_ptr(), ws.data_ptr(),
                           ws.numel(), stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(mx.strerror(rc))

    G = max(copies, min(128, calls_target // replays) // copies * copies)
    timer = GraphTimer(call, G, stream)
    timer.soak(0.4)
    wall0 = time.time()
    ms, per_call = timer.run(replays)
    wall1 = time.time()
    calls = replays * G
    us = ms * 1e3 / calls
    nbytes = ffn_chain_bytes(t, hidden, inter)
    peak, _ = hbm_peak()
    gbs = nbytes / (us * 1e-6) / 1e9
    two_launch = t <= 4 and hidden % 512 == 0 and inter % 512 == 0
    kernel = ("mxfp4::f4::f4_linear_kernel<npad, 0> (W1, fp32 a|b) then f4_linear_kernel<npad, 1> "
              "(W2, SiLU(a)*b converted in the kernel)" if two_launch else
              "mxfp4::ffn_chain_kernel (stream_body<FfnUp> then stream_body<FfnDown>, cooperative)")
    return {"us_per_call": round(us, 3), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
            "spread_us_per_call": percentiles(per_call), "calls": calls, "bytes_per_call": nbytes,
            "kernel": kernel, "launches_per_call": 2 if two_launch else 1,
            "memsets_per_call": 0 if two_launch else 1,
            "clocks": clocks.summary(wall0 - 0.5, wall1 + 0.1)}


_MOE_WEIGHTS = {}  # the expert weights, shared by the MoE runs of one bench process


def moe_weights(device, e, hidden, inter, seed):
    import torch

    import mxfp4_weight_streaming_gb300 as mx
    import synth
    w1q = torch.empty((e, 2 * inter, hidden // 2), dtype=torch.uint8, device=device)
    w1s = torch.empty((e, 2 * inter, hidden // 32), dtype=torch.uint8, device=device)
    w2q = torch.empty((e, hidden, inter // 2), dtype=torch.uint8, device=device)
    w2s = torch.empty((e, hidden, inter // 32), dtype=torch.uint8, device=device)
    for ex in range(e):
        a = synth.weights(seed, 2 * inter, hidden, device=device, row0=ex * 2 * inter)
        q, sc = mx.quantize(a)
        w1q[ex].copy_(q.view(2 * inter, -1))
        w1s[ex].copy_(sc.view(2 * inter, -1))
        b = synth.weights(seed, hidden, inter, tid=synth.TID_W2, device=device, row0=ex * hidden)
        q, sc = mx.quantize(b)
        w2q[ex].copy_(q.view(hidden, -1))
        w2s[ex].copy_(sc.view(hidden, -1))
        del a, b
    return w1q, w1s, w2q, w2s


def run_moe(steps: int, device, clocks, replays: int = 10, t: int | None = None):
    """Grouped top-8 MoE decode step (256 experts, T=32 unless t is given):
    one mxfp4_moe call per step; bytes = distinct routed experts' W1+W2 (+ x,
    logits, y)."""
    import torch

    import mxfp4_weight_streaming_gb300 as mx
    import synth

    m = MOE
    e, top_k, hidden, inter, seed = m["e"], m["top_k"], m["hidden"], m["inter"], m["seed"]
    t = m["t"] if t is None else t
    key = (str(device), e, hidden, inter, seed)
    if key not in _MOE_WEIGHTS:
        _MOE_WEIGHTS.clear()
        _MOE_WEIGHTS[key] = moe_weights(device, e, hidden, inter, seed)
    w1q, w1s, w2q, w2s = _MOE_WEIGHTS[key]
    x = synth.tokens(seed, t, hidden, device=device)
    lg = synth.logits(seed, t, e, device=device)
    distinct = int(torch.unique(torch.topk(lg.cpu(), top_k, dim=1).indices).numel())
    ws = mx.moe_workspace(t, e, top_k, hidden, inter, device)
    y = torch.empty((t, hidden), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device)
    lib = mx.load()
    args = [x.data_ptr(), t, hidden, lg.data_ptr(), e, top_k, w1q.data_ptr(), w1s.data_ptr(), w2q.data_ptr(),
            w2s.data_ptr(), inter, y.data_ptr(), None, None, ws.data_ptr(), ws.numel(), stream.cuda_stream]

    def call(i):
        rc = lib.mxfp4_moe(*args)
        if rc != 0:
            raise RuntimeError(mx.strerror(rc))

    G = max(1, min(steps // replays, 20))
    timer = GraphTimer(call, G, stream)
    timer.soak(0.5)
    wall0 = time.time()
    ms, per_call = timer.run(replays)
    wall1 = time.time()
    calls = replays * G
    us = ms * 1e3 / calls
    nbytes = distinct * moe_expert_bytes(hidden, inter) + 2 * t * hidden + 4 * t * e + 2 * t * hidden
    peak, _ = hbm_peak()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_call": round(us, 2), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
            "spread_us_per_call": percentiles(per_call), "calls": calls,
            "distinct_experts": distinct, "bytes_per_call": nbytes, "launches_per_call": 4,
            "kernel": "mxfp4::moe_route_kernel, stream_kernel<GateUpProblem>, stream_kernel<DownProblem>, "
                      "moe_combine_kernel",
            "timing": f"{replays} CUDA graph replays of {G} calls (4 kernels each), device events",
            "clocks": clocks.summary(wall0 - 0.6, wall1 + 0.1)}


# ------------------------------------------------------- CPU oracle timing
def cpu_baseline(wl_name: str, budget_s: float = 12.0):
    """The oracle, as it stands, on this host's cores, on a bounded sample:
    the workload's full call if it fits the budget, else a row subset scaled
    to the same metric (GB/s of the same algorithmic bytes)."""
    import numpy as np

    import oracle
    import synth

    wl = WORKLOADS[wl_name]
    t, k, n = wl["t"], wl["k"], wl["n"]
    rows = n
    # weights for the sampled rows only (CPU generation)
    probe = min(n, 512)
    w = synth.weights(wl["seed"], probe, k, x64_blocks=wl["x64"]).numpy()
    wq, ws = oracle.quantize(w)
    x = synth.tokens(wl["seed"], t, k)
    t0 = time.perf_counter()
    oracle.linear(x, wq, ws)
    dt = time.perf_counter() - t0
    per_row = dt / probe
    rows = int(min(n, max(probe, budget_s / max(per_row, 1e-9))))
    if rows > probe:
        w = synth.weights(wl["seed"], rows, k, x64_blocks=wl["x64"]).numpy()
        wq, ws = oracle.quantize(w)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.linear(x, wq, ws)
        reps += 1
        if time.perf_counter() - t0 > budget_s / 2 or reps >= 50:
            break
    dt = (time.perf_counter() - t0) / reps
    frac = rows / n
    bytes_sample = algorithmic_bytes(t, k, n) * frac
    gbs = bytes_sample / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} of {n} output rows, all {t} tokens, {reps} repetition(s); "
                      f"{dt * 1e3:.1f} ms per sample ({dt / frac * 1e3:.1f} ms per full call)"}


def run_reference(args, wl_name: str):
    """The reference arm: the CPU oracle timed on this host (no reference
    implementation exists to install); bounded so the run ends in minutes."""
    t_start = time.time()
    wl = WORKLOADS[wl_name]
    steps_budget = max(5.0, 60.0 / max(1, args.steps + args.warmup))
    cb = cpu_baseline(wl_name, budget_s=min(12.0, steps_budget))
    value = cb["value"]
    t, k, n = wl["t"], wl["k"], wl["n"]
    bytes_call = algorithmic_bytes(t, k, n)
    ms = bytes_call / (value * 1e9) * 1e3 if value > 0 else None
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": wl_name, "T": t, "K": k, "N": n, "bytes_per_call": bytes_call},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(time.time() - t_start, 2),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the headline workload (skip the other configurations)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, args.workload)), flush=True)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    import mxfp4_weight_streaming_gb300 as mx
    from mxfp4_weight_streaming_gb300 import build as b
    if rank == 0:
        b.build()
    if world > 1:
        torch.distributed.barrier()
    mx.load()
    # One clock sampler for the whole run, started before anything is timed
    # (nvidia-smi's start-up can stall the first CUDA launches after it);
    # each workload reads the samples of its own time window.
    clocks = ClockSampler(gpu_index())
    clocks.start()
    time.sleep(2.0)
    res = run_ours(args, args.workload, rank, world, device, with_cpu_baseline=(rank == 0 and world == 1
                                                                                 and not args.no_cpu_baseline),
                   clocks=clocks)
    if not args.no_workloads and rank == 0:
        # Every other configuration, timed on rank 0 (replicas: the same on every GPU).
        extra = {}
        cache = {}
        for name in WORKLOADS:
            if name == args.workload:
                continue
            try:
                extra[name] = measure_dense(name, device, cache, clocks)
            except Exception as ex:  # report, do not hide
                extra[name] = {"error": str(ex)[:300]}
            torch.cuda.empty_cache()
        cache.clear()
        torch.cuda.empty_cache()
        for name in FFN_CHAIN:
            try:
                extra[name] = measure_ffn_chain(name, device, clocks)
            except Exception as ex:
                extra[name] = {"error": str(ex)[:300]}
            torch.cuda.empty_cache()
        try:
            extra[MOE_WORKLOAD] = run_moe(200, device, clocks)
        except Exception as ex:
            extra[MOE_WORKLOAD] = {"error": str(ex)[:300]}
        torch.cuda.empty_cache()
        try:
            extra[f"moe_e256_top8_t{MOE_LARGE_T}"] = run_moe(100, device, clocks, t=MOE_LARGE_T)
        except Exception as ex:
            extra[f"moe_e256_top8_t{MOE_LARGE_T}"] = {"error": str(ex)[:300]}
        _MOE_WEIGHTS.clear()
        torch.cuda.empty_cache()
        res["workloads"] = extra
    clocks.stop()
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
