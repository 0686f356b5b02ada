#!/usr/bin/env python3
"""Benchmark of the fused attention forward (libfa) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

One step = one pass of the whole path over one batch of the workload, by
default the largest configuration the path is specified on that fits one GPU:
"Z=1 Hq=32 Hkv=8 (GQA group 4) Nq=Nkv=32768 D=128 bf16, causal" -- one fa_fwd
launch.  Metric: attention forward TFLOP/s, counting 4*Nq*Nkv*D per head and
half of it for causal.  Inputs are seeded synthetic N(0,1) (seeded_inputs);
input sets rotate so that consecutive steps never find their operands in L2.
Rank 0 prints one JSON line; besides the headline it times the Z=4 H=16
N=1024 D=128 workload and the D=128, N>=4096 non-causal shapes the
throughput target is stated on, each with its own clock record.

--profile runs only eager launches of --workload on one input set (for ncu).

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload (rows computed one by one).
N > 1 runs one independent replica per GPU ("replicas only": the path needs
no exchange between GPUs); value = all ranks' FLOPs / max time over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (causal-halved) and % of GB300 dense bf16/fp16 peak"
L2_BYTES = 129 * 2 ** 20

WORKLOADS = {
    # name: (Z, Hq, Hkv, Nq, Nkv, D, dtype, [causal flags per step])
    "z4_h16_n1024_d128_bf16": (4, 16, 16, 1024, 1024, 128, "bf16", [False, True]),
    "z1_hq32_hkv8_nq1024_nkv8192_d128_bf16_cross": (1, 32, 8, 1024, 8192, 128, "bf16", [False]),
    "z1_hq32_hkv8_n8192_d128_bf16_noncausal": (1, 32, 8, 8192, 8192, 128, "bf16", [False]),
    "z1_hq32_hkv8_n32768_d128_bf16_causal": (1, 32, 8, 32768, 32768, 128, "bf16", [True]),
    "z128_h8_n1024_d128_fp16": (128, 8, 8, 1024, 1024, 128, "fp16", [False, True]),
    "z128_h8_n1024_d64_fp16": (128, 8, 8, 1024, 1024, 64, "fp16", [False, True]),
    "z8_h16_n2048_d16_fp16": (8, 16, 16, 2048, 2048, 16, "fp16", [False, True]),
    "z8_h16_n2048_d32_fp16": (8, 16, 16, 2048, 2048, 32, "fp16", [False, True]),
    "z8_h16_n2048_d64_fp16": (8, 16, 16, 2048, 2048, 64, "fp16", [False, True]),
    "z8_h16_n2048_d128_bf16": (8, 16, 16, 2048, 2048, 128, "bf16", [False, True]),
    "z8_h16_n2048_d256_bf16": (8, 16, 16, 2048, 2048, 256, "bf16", [False, True]),
    "z1_h2_n128_d64_fp16_tiny": (1, 2, 2, 128, 128, 64, "fp16", [False]),
    # few query tiles against many keys: the shapes fa_fwd_splitkv is for
    "z1_hq32_hkv8_nq1_nkv32768_d128_bf16_decode": (1, 32, 8, 1, 32768, 128, "bf16", [False]),
    "z1_h8_nq128_nkv65536_d128_bf16": (1, 8, 8, 128, 65536, 128, "bf16", [False]),
}
MAIN = "z1_hq32_hkv8_n32768_d128_bf16_causal"
# the shapes the throughput target is stated on (D = 128, N >= 4096, non-causal)
TARGET_SHAPES = ["z1_hq32_hkv8_n8192_d128_bf16_noncausal", "z1_hq32_hkv8_nq1024_nkv8192_d128_bf16_cross"]
# timed besides the headline, each as its own line (rotated inputs, own clock record)
EXTRA_SHAPES = ["z4_h16_n1024_d128_bf16"] + TARGET_SHAPES
# timed through both entry points: whole tiles (fa_fwd) and cut key ranges where that pays (fa_fwd_splitkv)
SPLIT_SHAPES = ["z1_hq32_hkv8_nq1_nkv32768_d128_bf16_decode", "z1_h8_nq128_nkv65536_d128_bf16",
                "z1_hq32_hkv8_nq1024_nkv8192_d128_bf16_cross"]


def flops_of(Z, Hq, Nq, Nkv, D, causal) -> float:
    f = 4.0 * Z * Hq * Nq * Nkv * D
    return f / 2 if causal else f


def step_flops(wl) -> float:
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    return sum(flops_of(Z, Hq, Nq, Nkv, D, c) for c in flags)


def io_bytes(wl):
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    qkv = 2 * (Z * Hq * Nq * D + 2 * Z * Hkv * Nkv * D)
    out = len(flags) * (2 * Z * Hq * Nq * D + 4 * Z * Hq * Nq)
    return qkv, out


def algorithmic_bytes(wl) -> int:
    """Read Q, K, V once and write O and lse once (per launch)."""
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    return 2 * (2 * Z * Hq * Nq * D + 2 * Z * Hkv * Nkv * D) + 4 * Z * Hq * Nq


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# the sources the forward kernel of head dim D is compiled from
FWD_SOURCES = ["fa_fwd_kernel.cuh", "fa_fwd_chain_kernel.cuh", "fa_fwd_pair_kernel.cuh", "fa_ptx.cuh", "fa_params.h",
               "fa_launch.h", "fa_fwd_dim.cu"]


def kernel_source_hash() -> str:
    """Hash of the forward kernel's own sources (a change anywhere else leaves its counters valid)."""
    h = hashlib.sha256()
    for name in FWD_SOURCES:
        h.update(name.encode() + b"\0" + open(os.path.join(ROOT, "exact_attention_44_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(f"{kernel} {workload}")
    except Exception:
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def kernel_name(wl, causal) -> str:
    Z, Hq, Hkv, Nq, Nkv, D, dtype, _ = wl
    return f"fa_fwd_kernel<{D},{str(causal).lower()},{'bf16' if dtype == 'bf16' else 'fp16'}>"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ------------------------------------------------------------------ native --

def make_inputs(wl, seed, device):
    import torch

    import seeded_inputs as si
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    q, k, v = si.qkv(seed, Z, Hq, Hkv, Nq, Nkv, D, dtype)
    host = [si.as_torch(x, dtype).pin_memory() for x in (q, k, v)]
    return host, [h.to(device) for h in host]


def time_workload(fa, wl, steps, warmup, device, stream, world, eager=False, dev0=None, sample_clocks=True):
    """Time `steps` steps of a workload (every causal flag of it once per step).

    Input sets rotate so that their total exceeds 3x L2: no step finds its
    operands in L2 from the step before.  Unless eager, the timed loop replays
    CUDA graphs: per causal flag, one graph holding that flag's launch on each
    input set in turn; the K % nsets remaining steps run as eager launches.
    CUDA events on the launching stream bracket every replay; nvidia-smi
    samples the clocks meanwhile.  Returns a dict of timings."""
    import torch

    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    scale = 1.0 / math.sqrt(D)
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    per_set = sum(io_bytes(wl))
    nsets = max(2, min(8, math.ceil(3 * L2_BYTES / per_set)))
    if dev0 is None:
        _, dev0 = make_inputs(wl, 0, device)
    sets = [dev0] + [[x.clone() for x in dev0] for _ in range(nsets - 1)]
    outs = [[(torch.empty((Z, Hq, Nq, D), dtype=tdt, device=device),
              torch.empty((Z, Hq, Nq), dtype=torch.float32, device=device)) for _ in flags] for _ in range(nsets)]

    def launch(i, f):
        q, k, v = sets[i % nsets]
        o, lse = outs[i % nsets][f]
        fa.fa_fwd(q, k, v, o=o, lse=lse, scale=scale, causal=flags[f], stream=stream)

    for i in range(warmup):  # untimed warm-up steps
        for f in range(len(flags)):
            launch(i, f)
    torch.cuda.synchronize(device)
    code, word = fa.fa_device_status(stream)
    if code != fa.FA_OK:
        raise RuntimeError(f"device status after warm-up: {word:#x}")
    graphs = []
    if not eager:
        with torch.cuda.stream(stream):
            for f in range(len(flags)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(nsets):
                        launch(i, f)
                graphs.append(g)
        for g in graphs:
            g.replay()
        torch.cuda.synchronize(device)
    # exactly `steps` steps: steps // nsets replays of every flag's graph, then
    # the remaining steps as eager launches, all inside the timed region
    reps = steps // nsets if graphs else 0
    tail = steps - reps * nsets
    barrier(world)
    clocks = ClockSampler(device.index if device.index is not None else 0) if sample_clocks else None
    time.sleep(0.25 if clocks else 0)
    torch.cuda.synchronize(device)
    nrec = reps + tail
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(flags) + 1)] for _ in range(nrec)]
    for r in range(reps):
        for f in range(len(flags)):
            ev[r][f].record(stream)
            graphs[f].replay()
        ev[r][len(flags)].record(stream)
    for x in range(tail):
        e = ev[reps + x]
        for f in range(len(flags)):
            e[f].record(stream)
            launch(reps * nsets + x, f)
        e[len(flags)].record(stream)
    torch.cuda.synchronize(device)
    clock = clocks.stop() if clocks else None
    barrier(world)
    total_ms = ev[0][0].elapsed_time(ev[-1][-1])
    # per-launch durations: a graph replay holds nsets launches of its flag
    per_kernel_ms = [[ev[r][f].elapsed_time(ev[r][f + 1]) / nsets for r in range(reps) for _ in range(nsets)] +
                     [ev[reps + x][f].elapsed_time(ev[reps + x][f + 1]) for x in range(tail)]
                     for f in range(len(flags))]
    code, word = fa.fa_device_status(stream)
    if code != fa.FA_OK:
        raise RuntimeError(f"device status after timing: {word:#x}")
    launch_desc = ("eager fa_fwd calls" if not graphs else
                   f"CUDA graph per causal flag, {nsets} fa_fwd launches (one per input set) per replay")
    del sets, outs, graphs
    return {"total_ms": total_ms, "per_kernel_ms": per_kernel_ms, "nsets": nsets, "per_set": per_set,
            "clock": clock, "launch": launch_desc}


def roofline_of(wl, t, peaks, workload):
    """The dominant launch (largest share of the step) against the bf16 tensor peak."""
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    shares = [sum(x) for x in t["per_kernel_ms"]]
    dom = max(range(len(flags)), key=lambda f: shares[f])
    dom_ms = statistics.fmean(t["per_kernel_ms"][dom])
    achieved = flops_of(Z, Hq, Nq, Nkv, D, flags[dom]) / (dom_ms * 1e-3) / 1e12
    kname = kernel_name(wl, flags[dom])
    return {"bound": "tensor", "kernel": kname, "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
            "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
            "frac_of_sustained": (round(achieved / peaks["bf16_tflops_sustained"], 4)
                                  if peaks.get("bf16_tflops_sustained") else None),
            "traffic": recorded_traffic(kname, workload),
            "algorithmic_bytes": algorithmic_bytes(wl), "ms_per_launch": round(dom_ms, 5)}


def run_native(args, rank, world, device):
    import torch

    import exact_attention_44_gb300 as fa

    fa.build()
    fa.load()
    peaks = load_peaks()
    wl = WORKLOADS[args.workload]
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    scale = 1.0 / math.sqrt(D)
    # a stream of its own (CUDA graphs are not captured on the default stream),
    # made current so that every copy and launch below is ordered on it
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)

    host, dev0 = make_inputs(wl, 0, device)
    t = time_workload(fa, wl, args.steps, args.warmup, device, stream, world, eager=args.eager, dev0=dev0,
                      sample_clocks=rank == 0)
    max_ms = all_reduce_max(t["total_ms"], world, device)
    flops = step_flops(wl)
    value = world * flops * args.steps / (max_ms * 1e-3) / 1e12
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic (seeded N(0,1))",
        "config": {"workload": args.workload, "Z": Z, "Hq": Hq, "Hkv": Hkv, "Nq": Nq, "Nkv": Nkv, "D": D,
                   "causal_per_step": flags, "scale": scale, "layout": "BNSD contiguous",
                   "l2": f"{t['nsets']} rotating input sets ({t['nsets'] * t['per_set'] / 2**20:.0f} MiB > 3x L2)",
                   "launch": t["launch"], "parallelism": "replicas only" if world > 1 else "single GPU"},
        "frac_of_peak": round(value / world / peaks["bf16_tflops"], 4),
        "per_launch_ms": {f"causal={c}": round(statistics.fmean(t["per_kernel_ms"][f]), 5)
                          for f, c in enumerate(flags)},
        "roofline": roofline_of(wl, t, peaks, args.workload),
        "gpu_launches": len(flags) * args.steps,
        "clocks": t["clock"],
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, wl, host, flags, scale, device, stream, world)
        if rank == 0:
            result["e2e"]["host_link"] = measure_host_link(wl, host, device, stream)
    del host, dev0
    torch.cuda.empty_cache()
    if args.shapes and rank == 0:
        result["extra_shapes"] = [measure_extra(fa, name, device, stream, peaks, world) for name in EXTRA_SHAPES
                                  if name != args.workload]
        result["split_kv_shapes"] = [measure_shape(name, device, stream, peaks, impl=impl)
                                     for name in SPLIT_SHAPES for impl in ("fwd", "splitkv")]
        result["variant_shapes"] = [measure_variant(name, device, stream, peaks) for name in VARIANT_SHAPES]
        result["variant_shapes"] += [measure_variant(name, device, stream, peaks, bwd=True) for name in VARIANT_SHAPES]
        result["bwd_shapes"] = [r for name in BWD_SHAPES for r in measure_bwd(name, device, stream, peaks)]
    return result


def measure_extra(fa, name, device, stream, peaks, world):
    """One more workload timed like the headline (graph replays, rotated inputs, own clock record)."""
    import torch

    wl = WORKLOADS[name]
    # about a quarter of a second of timed work
    steps = max(20, min(2000, int(0.25 / max(step_flops(wl) / 1.2e15, 1e-6))))
    t = time_workload(fa, wl, steps, 5, device, stream, world)
    value = step_flops(wl) * steps / (t["total_ms"] * 1e-3) / 1e12
    flags = wl[7]
    torch.cuda.empty_cache()
    return {"workload": name, "tflops": round(value, 2), "frac_of_peak": round(value / peaks["bf16_tflops"], 4),
            "ms_per_step": round(t["total_ms"] / steps, 5), "steps": steps,
            "per_launch_ms": {f"causal={c}": round(statistics.fmean(t["per_kernel_ms"][f]), 5)
                              for f, c in enumerate(flags)},
            "roofline": roofline_of(wl, t, peaks, name),
            "l2": f"{t['nsets']} rotating input sets", "launch": t["launch"], "clocks": t["clock"]}


def run_e2e(args, wl, host, flags, scale, device, stream, world):
    """Same metric through the public API with host buffers: H2D of Q/K/V from pinned memory,
    every launch of the step, D2H of O and lse, every step, all inside the timed region.

    Steps alternate between two streams, each with its own device and pinned host buffers,
    so that one step's device-to-host copies overlap the next step's host-to-device copies
    (opposite directions, separate copy engines); every step still moves all of its bytes.
    Events around each step's launches give the kernels' own time inside the loop (a step's
    launches start once its copies are in and the previous step's launches are done), and
    nvidia-smi samples the clocks over the loop."""
    import torch

    import exact_attention_44_gb300 as fa
    Z, Hq, Hkv, Nq, Nkv, D, dtype, _ = wl
    tdt = host[0].dtype
    streams = [stream, torch.cuda.Stream(device=device)]
    lanes = []
    for _ in streams:
        dev_in = [torch.empty_like(h, device=device) for h in host]
        outs = [(torch.empty((Z, Hq, Nq, D), dtype=tdt, device=device),
                 torch.empty((Z, Hq, Nq), dtype=torch.float32, device=device)) for _ in flags]
        host_out = [(torch.empty((Z, Hq, Nq, D), dtype=tdt).pin_memory(),
                     torch.empty((Z, Hq, Nq), dtype=torch.float32).pin_memory()) for _ in flags]
        lanes.append((dev_in, outs, host_out))
    steps = max(3, min(args.steps, 50))

    def step(i, spans=None):
        s = streams[i % 2]
        dev_in, outs, host_out = lanes[i % 2]
        with torch.cuda.stream(s):
            for d, h in zip(dev_in, host):
                d.copy_(h, non_blocking=True)
            if spans is not None:
                spans.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                spans[-1][0].record(s)
            for (o, lse), causal in zip(outs, flags):
                fa.fa_fwd(*dev_in, o=o, lse=lse, scale=scale, causal=causal, stream=s)
            if spans is not None:
                spans[-1][1].record(s)
            for (o, lse), (ho, hl) in zip(outs, host_out):
                ho.copy_(o, non_blocking=True)
                hl.copy_(lse, non_blocking=True)

    for i in range(4):
        step(i)
    torch.cuda.synchronize(device)
    barrier(world)
    clocks = ClockSampler(device.index if device.index is not None else 0) if int(os.environ.get("RANK", "0")) == 0 else None
    spans = []
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    streams[1].wait_event(a)
    for i in range(steps):
        step(i, spans)
    done = torch.cuda.Event()
    done.record(streams[1])
    stream.wait_event(done)
    b.record(stream)
    torch.cuda.synchronize(device)
    clock = clocks.stop() if clocks is not None else None
    ms = all_reduce_max(a.elapsed_time(b), world, device)
    # a step's launches run from when its copies are in and the previous step's are done
    ends = [a.elapsed_time(e1) for _, e1 in spans]
    kernel_ms = [ends[i] - max(a.elapsed_time(e0), ends[i - 1] if i else 0.0) for i, (e0, _) in enumerate(spans)]
    h2d, d2h = io_bytes(wl)
    del lanes
    out = {"value": round(world * step_flops(wl) * steps / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
           "ms_per_step": round(ms / steps, 4), "streams": 2,
           "kernel_ms_per_step": {"mean": round(statistics.fmean(kernel_ms), 4),
                                  "first": round(kernel_ms[0], 4), "last": round(kernel_ms[-1], 4)},
           "kernel_share": round(sum(kernel_ms) / ms, 4)}
    if clock is not None:
        out["clocks"] = clock
    return out


def measure_host_link(wl, host, device, stream, reps=10):
    """Plain pinned-memory copy bandwidth with the e2e step's byte counts: the host link's ceiling
    for e2e.  H2D of Q, K, V alone; D2H of O and lse alone; and both at once on two streams."""
    import torch

    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    dev_in = [torch.empty_like(h, device=device) for h in host]
    dev_out = [torch.empty((Z, Hq, Nq, D), dtype=host[0].dtype, device=device),
               torch.empty((Z, Hq, Nq), dtype=torch.float32, device=device)]
    host_out = [torch.empty_like(d, device="cpu").pin_memory() for d in dev_out]
    s2 = torch.cuda.Stream(device=device)
    h2d, d2h = io_bytes(wl)
    d2h = d2h // max(1, len(flags))  # one launch's outputs

    def timed(fn):
        fn()
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s2.wait_event(a)
        for _ in range(reps):
            fn()
        done = torch.cuda.Event()
        done.record(s2)
        stream.wait_event(done)
        b.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / reps

    def up():
        with torch.cuda.stream(stream):
            for d, h in zip(dev_in, host):
                d.copy_(h, non_blocking=True)

    def down(s=None):
        with torch.cuda.stream(s or stream):
            for d, h in zip(dev_out, host_out):
                h.copy_(d, non_blocking=True)

    ms_up = timed(up)
    ms_down = timed(down)
    ms_both = timed(lambda: (up(), down(s2)))
    del dev_in, dev_out, host_out
    return {"h2d_gbs": round(h2d / (ms_up * 1e-3) / 1e9, 1), "d2h_gbs": round(d2h / (ms_down * 1e-3) / 1e9, 1),
            "both_ms": round(ms_both, 4), "h2d_ms": round(ms_up, 4), "d2h_ms": round(ms_down, 4),
            "what": "plain pinned cudaMemcpyAsync of one step's inputs (H2D) and one launch's outputs (D2H), "
                    "alone and at once on two streams"}


def run_profile(args, device):
    """Eager launches of one workload on one input set, nothing else (a small, predictable ncu target)."""
    import torch

    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()
    wl = WORKLOADS[args.workload]
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    fa.fa_debug_force_chains(args.force_chains)
    _, (q, k, v) = make_inputs(wl, 0, device)
    stream = torch.cuda.current_stream(device)
    o = torch.empty((Z, Hq, Nq, D), dtype=q.dtype, device=device)
    lse = torch.empty((Z, Hq, Nq), dtype=torch.float32, device=device)
    ws = fa.workspace_for(D, device) if args.profile_impl == "splitkv" else None
    for _ in range(args.warmup + args.steps):
        for c in flags:
            if ws is not None:
                fa.fa_fwd_splitkv(q, k, v, o=o, lse=lse, causal=c, workspace=ws, stream=stream)
            else:
                fa.fa_fwd(q, k, v, o=o, lse=lse, causal=c, stream=stream)
    torch.cuda.synchronize(device)
    code, word = fa.fa_device_status(stream)
    if code != fa.FA_OK:
        raise RuntimeError(f"device status: {word:#x}")
    print(json.dumps({"profile": args.workload, "launches": (args.warmup + args.steps) * len(flags)}), flush=True)


def measure_shape(name, device, stream, peaks, steps=10, impl="fwd"):
    """TFLOP/s of one extra workload (eager launches, 10 steps, inputs > L2 or rotated).

    impl "fwd" calls fa_fwd; "splitkv" calls fa_fwd_splitkv, which cuts the key
    ranges across SMs when that beats whole tiles."""
    import torch

    import exact_attention_44_gb300 as fa
    wl = WORKLOADS[name]
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    scale = 1.0 / math.sqrt(D)
    per_set = sum(io_bytes(wl))
    nsets = max(1, min(6, math.ceil(3 * L2_BYTES / per_set)))
    _, dev0 = make_inputs(wl, 0, device)
    sets = [dev0] + [[x.clone() for x in dev0] for _ in range(nsets - 1)]
    o = torch.empty((Z, Hq, Nq, D), dtype=dev0[0].dtype, device=device)
    lse = torch.empty((Z, Hq, Nq), dtype=torch.float32, device=device)
    ws = fa.workspace_for(D, device) if impl == "splitkv" else None

    def call(i, c):
        if impl == "splitkv":
            fa.fa_fwd_splitkv(*sets[i % nsets], o=o, lse=lse, scale=scale, causal=c, workspace=ws, stream=stream)
        else:
            fa.fa_fwd(*sets[i % nsets], o=o, lse=lse, scale=scale, causal=c, stream=stream)

    for i in range(3):
        for c in flags:
            call(i, c)
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        for c in flags:
            call(i, c)
    b.record(stream)
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / steps
    tf = step_flops(wl) / (ms * 1e-3) / 1e12
    code, word = fa.fa_device_status(stream)
    if code != fa.FA_OK:
        raise RuntimeError(f"device status after {name}: {word:#x}")
    del sets, dev0, ws
    torch.cuda.empty_cache()
    return {"workload": name, "impl": impl, "tflops": round(tf, 2), "frac_of_peak": round(tf / peaks["bf16_tflops"], 4),
            "ms_per_step": round(ms, 4), "steps": steps}


# fa_fwd_ex workloads: name -> (Z, Hq, Hkv, N, D, dtype, causal, window, alibi, varlen lengths or None)
VARIANT_SHAPES = {
    "z4_h16_n4096_d128_bf16_causal_window512": (4, 16, 16, 4096, 128, "bf16", True, (512, 0), False, None),
    "z4_h16_n2048_d128_bf16_causal_alibi": (4, 16, 16, 2048, 128, "bf16", True, (-1, -1), True, None),
    "varlen_16seq_256to4096_h16_d128_bf16_causal": (16, 16, 16, 0, 128, "bf16", True, (-1, -1), False, "seeded"),
    "z2_h16_n4096_d256_bf16_causal_window512": (2, 16, 16, 4096, 256, "bf16", True, (512, 0), False, None),
}


def variant_lengths(Z, seed=0):
    """Seeded sequence lengths, uniform on [256, 4096]."""
    import numpy as np
    return np.random.default_rng(seed).integers(256, 4097, size=Z)


def variant_flops(Z, Hq, N, D, causal, window, lens):
    """4 D per kept (query, key) pair; causal without a window counts half of N^2, as the metric does."""
    if lens is not None:
        return sum(4.0 * Hq * L * L * D / (2 if causal else 1) for L in lens)
    wl, wr = window
    if wl < 0 and wr < 0:
        return flops_of(Z, Hq, N, N, D, causal)
    pairs = 0
    for i in range(N):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = N - 1 if wr < 0 else min(N - 1, i + wr)
        if causal:
            hi = min(hi, i)
        pairs += max(0, hi - lo + 1)
    return 4.0 * Z * Hq * pairs * D


def measure_variant(name, device, stream, peaks, steps=10, bwd=False):
    """TFLOP/s of fa_fwd_ex on a window / ALiBi / variable-length workload (kept pairs only); with bwd,
    of fa_bwd_ex on it (5 products of the kept pairs)."""
    import numpy as np
    import torch

    import exact_attention_44_gb300 as fa
    import seeded_inputs as si
    Z, Hq, Hkv, N, D, dtype, causal, window, alibi, varlen = VARIANT_SHAPES[name]
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    lens = variant_lengths(Z) if varlen else None
    kw = {}
    if lens is not None:
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        total = int(cu[-1])
        shape_q, shape_k = (1, Hq, total, D), (1, Hkv, total, D)
        cu_t = torch.from_numpy(cu).to(device)
        kw.update(cu_seqlens_q=cu_t, cu_seqlens_k=cu_t, max_seqlen_q=int(lens.max()))
        bwd_kw = dict(cu_seqlens_q=cu_t, cu_seqlens_k=cu_t, max_seqlen_q=int(lens.max()), max_seqlen_k=int(lens.max()))
    else:
        shape_q, shape_k = (Z, Hq, N, D), (Z, Hkv, N, D)
        bwd_kw = {}
    nq, nk = int(np.prod(shape_q)), int(np.prod(shape_k))
    q = si.as_torch(si.normals(0, 0, nq, dtype).reshape(shape_q), dtype).to(device)
    k = si.as_torch(si.normals(0, nq, nk, dtype).reshape(shape_k), dtype).to(device)
    v = si.as_torch(si.normals(0, nq + nk, nk, dtype).reshape(shape_k), dtype).to(device)
    if alibi:
        kw["alibi_slopes"] = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32,
                                          device=device)
    o = torch.empty_like(q)

    def call():
        fa.fa_fwd_ex(q, k, v, o=o, causal=causal, window=window, stream=stream, **kw)

    if bwd:
        o, lse = fa.fa_fwd_ex(q, k, v, causal=causal, window=window, stream=stream, **kw)
        do = si.as_torch(si.normals(1, 0, nq, dtype).reshape(shape_q), dtype).to(device)
        rows = int(lens.max()) if lens is not None else N  # packed: rows of the longest sequence
        ws = torch.empty(fa.fa_bwd_workspace_size(Z, Hq, rows, D), dtype=torch.uint8, device=device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        slopes = kw.get("alibi_slopes")

        def call():  # noqa: F811 (the timed call of this mode)
            fa.fa_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, causal=causal, window=window, alibi_slopes=slopes,
                         workspace=ws, stream=stream, **bwd_kw)

    for _ in range(3):
        call()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        call()
    b.record(stream)
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / steps
    code, word = fa.fa_device_status(stream)
    if code != fa.FA_OK:
        raise RuntimeError(f"device status after {name}: {word:#x}")
    tf = (2.5 if bwd else 1.0) * variant_flops(Z, Hq, N, D, causal, window, lens) / (ms * 1e-3) / 1e12
    return {"workload": name, "impl": "bwd_ex" if bwd else "fwd_ex", "tflops": round(tf, 2),
            "frac_of_peak": round(tf / peaks["bf16_tflops"], 4), "ms_per_step": round(ms, 4), "steps": steps,
            "flops": "kept (query, key) pairs x 10 D (5 products)" if bwd else "kept (query, key) pairs x 4 D"}


# fa_bwd workloads (gradients of the forward; 5 products of 2 N^2 D per head, half for causal)
BWD_SHAPES = ["z4_h16_n1024_d128_bf16", "z1_hq32_hkv8_n8192_d128_bf16_noncausal", "z8_h16_n2048_d64_fp16",
              "z8_h16_n2048_d256_bf16", "z1_hq32_hkv8_n32768_d128_bf16_causal"]


def measure_bwd(name, device, stream, peaks, steps=10):
    """TFLOP/s of fa_bwd (all three of its kernels) per causal flag of a workload."""
    import torch

    import exact_attention_44_gb300 as fa
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = WORKLOADS[name]
    _, dev0 = make_inputs(WORKLOADS[name], 0, device)
    q, k, v = dev0
    do = torch.randn_like(q)
    ws = torch.empty(fa.fa_bwd_workspace_size(Z, Hq, Nq, D), dtype=torch.uint8, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    out = []
    for causal in flags:
        o, lse = fa.fa_fwd(q, k, v, causal=causal, stream=stream)

        def call():
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal=causal, workspace=ws, stream=stream)

        for _ in range(3):
            call()
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            call()
        b.record(stream)
        torch.cuda.synchronize(device)
        ms = a.elapsed_time(b) / steps
        code, word = fa.fa_device_status(stream)
        if code != fa.FA_OK:
            raise RuntimeError(f"device status after the backward of {name}: {word:#x}")
        tf = 2.5 * flops_of(Z, Hq, Nq, Nkv, D, causal) / (ms * 1e-3) / 1e12
        out.append({"workload": name, "causal": causal, "impl": "bwd", "tflops": round(tf, 2),
                    "frac_of_peak": round(tf / peaks["bf16_tflops"], 4), "ms_per_step": round(ms, 4), "steps": steps,
                    "flops": "10 N^2 D per head (5 products), half for causal"})
    del dev0, q, k, v, do, ws, dq, dk, dv
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ oracle --

def run_oracle_sample(wl, budget_s: float):
    """Time the fp64 CPU oracle on rows of the workload, growing the sample until ~budget_s."""
    import numpy as np

    import oracle
    import seeded_inputs as si
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    scale = 1.0 / math.sqrt(D)
    # one GQA group of (z = 0, kv head 0): its query heads and K/V
    g = Hq // Hkv
    nq = g * Nq * D
    q = si.normals(0, 0, nq, dtype).reshape(1, g, Nq, D)  # BNSD: the first g heads of z = 0
    k = si.normals(0, Z * Hq * Nq * D, Nkv * D, dtype).reshape(1, 1, Nkv, D)
    v = si.normals(0, Z * Hq * Nq * D + Z * Hkv * Nkv * D, Nkv * D, dtype).reshape(1, 1, Nkv, D)
    threads = oracle.host_threads()
    rng = np.random.default_rng(0)
    rows_n, elapsed, done_flops = 16, 0.0, 0.0
    total_rows = 0
    while True:
        rows = np.sort(rng.integers(0, g * Nq, size=rows_n)).astype(np.int64)
        f = 0.0
        for c in flags:
            kept = (rows % Nq + 1).clip(max=Nkv) if c else np.full(rows.shape, Nkv)
            f += float(np.sum(4.0 * kept * D))
        t0 = time.perf_counter()
        for c in flags:
            oracle.attention_fwd(q, k, v, dtype, scale, c, rows=rows, nthreads=threads)
        dt = time.perf_counter() - t0
        elapsed += dt
        done_flops += f
        total_rows += rows_n
        if elapsed >= budget_s or dt > budget_s / 3:
            break
        rows_n *= 2
    return {"value": done_flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{total_rows} query rows of (z=0, kv head 0) of {WORKLOADS_NAME(wl)}, each for "
                      f"{'+'.join('causal' if c else 'non-causal' for c in flags)}, fp64, {elapsed:.1f} s"}


def WORKLOADS_NAME(wl):
    for k, v in WORKLOADS.items():
        if v == wl:
            return k
    return "workload"


def run_reference(args, rank, world):
    wl = WORKLOADS[args.workload]
    Z, Hq, Hkv, Nq, Nkv, D, dtype, flags = wl
    times, values = [], []
    budget = max(0.05, min(args.cpu_budget, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        run_oracle_sample(wl, budget / 4)
    info = None
    for i in range(args.steps):
        info = run_oracle_sample(wl, budget)
        values.append(info["value"])
    value = statistics.fmean(values)
    ms_per_step = step_flops(wl) / (value * 1e12) * 1e3  # time the oracle would take for one whole step
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1))",
            "config": {"workload": args.workload, "Z": Z, "Hq": Hq, "Hkv": Hkv, "Nq": Nq, "Nkv": Nkv, "D": D,
                       "causal_per_step": flags, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": info["cores"], "kind": "oracle",
                             "sample": info["sample"]},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ------------------------------------------------------------------ dist ----

def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _cuda_ok() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=MAIN)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager fa_fwd calls instead of CUDA-graph replays")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shapes", dest="shapes", action="store_true", default=True,
                    help="also time the Z=4 H=16 N=1024 workload, the D=128 N>=4096 non-causal target shapes, "
                         "split-KV, variant and backward workloads (default)")
    ap.add_argument("--no-shapes", dest="shapes", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for cpu_baseline (and the cap per step of --impl reference)")
    ap.add_argument("--profile", action="store_true",
                    help="only W + K eager launches of --workload on one input set, no timing (an ncu target)")
    ap.add_argument("--profile-impl", choices=["fwd", "splitkv"], default="fwd",
                    help="with --profile: the entry point launched (fa_fwd or fa_fwd_splitkv)")
    ap.add_argument("--force-chains", type=int, choices=[0, 1, 2], default=0,
                    help="with --profile: 0 the library's choice, 1 two softmax chains, 2 one")
    ap.add_argument("--bwd-only", action="store_true",
                    help="time only fa_bwd on --workload (one JSON line per causal flag; for profiling)")
    ap.add_argument("--all", action="store_true",
                    help="instead of the bench line, time every workload (one JSON line each) for the results table")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "native":
        ap.error("--warmup must be >= 3")
    rank, world, local = init_dist()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the native path has no CPU fallback)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.profile:
        run_profile(args, device)
        return 0
    if args.bwd_only:
        import exact_attention_44_gb300 as fa
        fa.build()
        fa.load()
        for r in measure_bwd(args.workload, device, torch.cuda.current_stream(device), load_peaks(), steps=args.steps):
            print(json.dumps(r), flush=True)
        return 0
    if args.all:
        import exact_attention_44_gb300 as fa
        fa.build()
        fa.load()
        peaks = load_peaks()
        for name, wl in list(WORKLOADS.items()):
            for causal in wl[7]:
                single = wl[:7] + ([causal],)
                WORKLOADS[name + ("_causal" if causal else "_noncausal")] = single
                for impl in ("fwd", "splitkv"):
                    r = measure_shape(name + ("_causal" if causal else "_noncausal"), device,
                                      torch.cuda.current_stream(device), peaks, steps=20, impl=impl)
                    r.update(dtype=wl[6], causal=causal)
                    print(json.dumps(r), flush=True)
        return 0
    result = run_native(args, rank, world, device)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = run_oracle_sample(WORKLOADS[args.workload], args.cpu_budget)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
