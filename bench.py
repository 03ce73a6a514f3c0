"""Benchmark of the W4A16 layer on one GB300 (or N replicas under torchrun).

A step is one decode pass over L layers (32 by default): L launches of the
GEMV, each on its own copy of the packed weights (so every launch streams its
weights from HBM, not L2), replayed as one CUDA graph. The headline workload is the gate_up-like decode GEMV
1 x 43008 x 5376, g=32, fp16, asymmetric; the same run also times the prefill
GEMM 2048 x 43008 x 5376, g=32, bf16 ("prefill" object).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --configs      # every named workload: median and min us per call

Prints one JSON line on rank 0. `value` is the whole-job GB/s over all ranks
(algorithmic bytes: packed weights + scales + packed zero-points + x + y).
`--impl reference` times the CPU FP64 oracle instead, on a bounded sample of
the same workload, and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w4a16_inputs import MX_WORKLOADS, WORKLOADS  # noqa: E402
from weight_only_int4_gb300.accounting import (dequant_bytes, layer_bytes, layer_flops, mx_dequant_bytes,  # noqa: E402
                                               mx_layer_bytes)

METRIC = "W4A16 GEMM GB/s (% of HBM peak) at M=1-4; TFLOP/s (% bf16 peak) at M=2048"
DECODE = "gemv_1x43008x5376_g32_f16_asym"
PREFILL = "gemm_2048x43008x5376_g32_bf16_asym"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
KERNEL_SOURCES = {
    "gemv": os.path.join(ROOT, "weight_only_int4_gb300", "csrc", "gemv.cu"),
    "gemm": os.path.join(ROOT, "weight_only_int4_gb300", "csrc", "gemm.cu"),
}


def code_hash(text: str) -> str:
    """sha256[:16] of a CUDA source with its comments and blank lines removed:
    edits to comments do not invalidate counters taken on the same code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    code = "\n".join(line.rstrip() for line in text.split("\n") if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def kernel_hash(kind: str) -> str:
    with open(KERNEL_SOURCES[kind], encoding="utf-8") as f:
        return code_hash(f.read())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t[workload]
        if e.get("kernel_sha256_16") != kernel_hash(kind):
            return None
        return int(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="w4a16_clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [v for v in sm if smax and v > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def _to_dev(a, act, torch):
    if act == "f16":
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


class Layer:
    """One workload on the device with `copies` independent weight sets."""

    def __init__(self, name, copies, torch, w4):
        self.wl = WORKLOADS[name]
        wl = self.wl
        case = wl.case(seed=0)
        self.x = _to_dev(case.x, wl.act, torch)
        s = _to_dev(case.s, wl.act, torch)
        q8 = torch.from_numpy(case.q).cuda()
        qw = w4.pack(q8, dim=0)
        del q8
        qz = None if case.z is None else w4.pack(torch.from_numpy(case.z).cuda(), dim=1)
        self.weights = [(qw, s, qz)] + [(qw.clone(), s.clone(), None if qz is None else qz.clone())
                                        for _ in range(copies - 1)]
        self.fn = getattr(w4, wl.kernel)
        if wl.kernel == "dequant":
            self.y = [torch.empty((wl.K, wl.N), dtype=self.x.dtype, device="cuda") for _ in range(copies)]
            self.ws = None
            self.bytes = dequant_bytes(wl.N, wl.K, wl.g, wl.symmetric, wl.act)
            self.flops = 0
            return
        self.y = [torch.empty((wl.M, wl.N), dtype=self.x.dtype, device="cuda") for _ in range(copies)]
        op = w4.OP_GEMV if wl.kernel == "gemv" else w4.OP_GEMM
        nws = w4.workspace_bytes(op, wl.M, wl.N, wl.K, wl.g)
        self.ws = w4.new_workspace(nws) if nws else None
        self.bytes = layer_bytes(wl.M, wl.N, wl.K, wl.g, wl.symmetric, wl.act)
        self.flops = layer_flops(wl.M, wl.N, wl.K)

    def step(self, x=None):
        if self.wl.kernel == "dequant":
            for (qw, s, qz), y in zip(self.weights, self.y):
                self.fn(qw, s, qz, self.wl.g, out=y)
            return
        x = self.x if x is None else x
        for (qw, s, qz), y in zip(self.weights, self.y):
            self.fn(x, qw, s, qz, self.wl.g, out=y, workspace=self.ws)


class MxLayer:
    """One MXFP4 workload (E2M1 codes, E8M0 exponents) with `copies` weight sets."""

    def __init__(self, name, copies, torch, w4):
        self.wl = wl = MX_WORKLOADS[name]
        case = wl.case(seed=0)
        self.x = _to_dev(case.x, "bf16", torch)
        q8 = torch.from_numpy(case.q).cuda()
        qw = w4.pack(q8, dim=0)
        del q8
        e = torch.from_numpy(case.e).cuda()
        self.weights = [(qw, e)] + [(qw.clone(), e.clone()) for _ in range(copies - 1)]
        self.fn = getattr(w4, "mxfp4_" + wl.kernel)
        self.ws = None
        if wl.kernel == "dequant":
            self.y = [torch.empty((wl.K, wl.N), dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
            self.bytes = mx_dequant_bytes(wl.N, wl.K)
            self.flops = 0
            return
        self.y = [torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
        op = w4.OP_GEMV if wl.kernel == "gemv" else w4.OP_GEMM
        nws = w4.workspace_bytes(op, wl.M, wl.N, wl.K, 32)
        self.ws = w4.new_workspace(nws) if nws else None
        self.bytes = mx_layer_bytes(wl.M, wl.N, wl.K)
        self.flops = layer_flops(wl.M, wl.N, wl.K)

    def step(self, x=None):
        x = self.x if x is None else x
        for (qw, e), y in zip(self.weights, self.y):
            if self.wl.kernel == "dequant":
                self.fn(qw, e, out=y)
            else:
                self.fn(x, qw, e, out=y, workspace=self.ws)


def time_graph(layer, steps, warmup, torch, barrier, per_step=None):
    """Device time of `steps` replays of a CUDA graph of one step (events on the
    replay stream). An event follows every replay, so `per_step` (a list, if
    given) receives each replay's own time; their sum is the total returned."""
    stream = torch.cuda.Stream()
    for _ in range(max(1, warmup)):
        layer.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer.step()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            g.replay()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    if per_step is not None:
        per_step.extend(ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(steps))
    return ev[0].elapsed_time(ev[steps]) / 1e3   # seconds


def time_graph_samples(layer, steps, warmup, torch):
    """Per-replay device times (seconds) of a CUDA graph of one step."""
    stream = torch.cuda.Stream()
    for _ in range(max(1, warmup)):
        layer.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer.step()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            e0.record(stream)
            g.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) / 1e3 for e0, e1 in ev]


def run_configs(args):
    """Every named workload on one GPU: median and min time per call over
    `steps` replays of a graph of L calls on distinct weight copies (L chosen so
    one replay streams >= 4x L2), GB/s of algorithmic bytes, TFLOP/s, and the
    fractions of the measured peaks."""
    import torch

    import weight_only_int4_gb300 as w4
    w4.load_library()
    torch.cuda.set_device(0)
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 128 << 20)
    peaks, peak_src = load_peaks()
    rows = []
    copy_gbs = box_copy_gbs(torch)
    clocks = ClockSampler(0)
    clocks.start()
    for name, wl in WORKLOADS.items():
        if args.match and args.match not in name:
            continue
        per = (dequant_bytes(wl.N, wl.K, wl.g, wl.symmetric, wl.act) if wl.kernel == "dequant" else
               layer_bytes(wl.M, wl.N, wl.K, wl.g, wl.symmetric, wl.act)).total
        L = copies_for(per, l2) if wl.kernel != "gemm" else 2
        layer = Layer(name, L, torch, w4)
        steps = max(5, args.steps if wl.kernel != "gemm" else args.steps // 10)
        t = [x / L for x in time_graph_samples(layer, steps, max(3, args.warmup), torch)]
        med, mn = statistics.median(t), min(t)
        rows.append({"workload": name, "kernel": wl.kernel, "calls_per_replay": L, "replays": steps,
                     "us_median": round(med * 1e6, 3), "us_min": round(mn * 1e6, 3),
                     "GBs": round(per / med / 1e9, 1), "TFLOPs": round(layer.flops / med / 1e12, 2),
                     "frac_hbm": round(per / med / 1e9 / peaks["hbm_gbs"], 4),
                     "frac_bf16": round(layer.flops / med / 1e12 / peaks["bf16_tflops"], 4)})
        del layer
        torch.cuda.empty_cache()
    for name, wl in MX_WORKLOADS.items():
        if args.match and args.match not in name:
            continue
        per = (mx_dequant_bytes(wl.N, wl.K) if wl.kernel == "dequant" else mx_layer_bytes(wl.M, wl.N, wl.K)).total
        L = copies_for(per, l2) if wl.kernel != "gemm" else 2
        layer = MxLayer(name, L, torch, w4)
        steps = max(5, args.steps if wl.kernel != "gemm" else args.steps // 10)
        t = [x / L for x in time_graph_samples(layer, steps, max(3, args.warmup), torch)]
        med, mn = statistics.median(t), min(t)
        rows.append({"workload": name, "kernel": "mxfp4_" + wl.kernel, "calls_per_replay": L, "replays": steps,
                     "us_median": round(med * 1e6, 3), "us_min": round(mn * 1e6, 3),
                     "GBs": round(per / med / 1e9, 1), "TFLOPs": round(layer.flops / med / 1e12, 2),
                     "frac_hbm": round(per / med / 1e9 / peaks["hbm_gbs"], 4),
                     "frac_bf16": round(layer.flops / med / 1e12 / peaks["bf16_tflops"], 4)})
        del layer
        torch.cuda.empty_cache()
    clk = clocks.stop()
    if w4.device_status() != w4.OK:
        raise RuntimeError("device-side error status after the timed region")
    return {"configs": rows, "peaks": peaks, "peak_source": peak_src, "clocks": clk,
            "this_gpu_copy_gbs": copy_gbs,
            "timing": "per-replay CUDA events around a CUDA graph of L calls; per call = replay / L"}


def time_e2e(layer, steps, warmup, torch):
    """Wall time of `steps` steps through the public API with host buffers:
    pinned x -> device, L calls, every y -> pinned host."""
    x_host = layer.x.cpu().pin_memory()
    y_host = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in layer.y]
    x_dev = torch.empty_like(layer.x)

    def one():
        x_dev.copy_(x_host, non_blocking=True)
        layer.step(x_dev)
        for yh, yd in zip(y_host, layer.y):
            yh.copy_(yd, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    h2d = x_host.numel() * x_host.element_size()
    d2h = sum(y.numel() * y.element_size() for y in y_host)
    return dt, h2d, d2h


def box_copy_gbs(torch, nbytes=1 << 30, reps=5):
    """Device-to-device copy bandwidth of this GPU (bytes read + written per
    second): context for the roofline, which is taken against the measured
    peak. GB300s of one pool differ by several per cent here."""
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    for _ in range(2):
        dst.copy_(src)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        dst.copy_(src)
    e1.record()
    torch.cuda.synchronize()
    gbs = 2 * nbytes * reps / (e0.elapsed_time(e1) / 1e3) / 1e9
    del src, dst
    torch.cuda.empty_cache()
    return round(gbs, 1)


# The decode workloads the metric names beside the headline (M = 1-4): the
# 1x2048x2048 g=128 case, the M = 4 g=128 sweep in fp16 and bf16, and the
# qkv-like and down-like shapes, symmetric and asymmetric.
METRIC_CONFIGS = [
    "gemv_1x2048x2048_g128_f16_asym",
    "gemv_4x2048x2048_g128_f16_asym", "gemv_4x2048x2560_g128_f16_asym",
    "gemv_4x6144x2048_g128_f16_asym", "gemv_4x4096x2048_g128_f16_asym",
    "gemv_4x2048x2048_g128_bf16_asym", "gemv_4x2048x2560_g128_bf16_asym",
    "gemv_4x6144x2048_g128_bf16_asym", "gemv_4x4096x2048_g128_bf16_asym",
    "gemv_1x16384x5376_g32_bf16_sym", "gemv_1x16384x5376_g32_bf16_asym",
    "gemv_1x5376x21504_g32_bf16_sym", "gemv_1x5376x21504_g32_bf16_asym",
]
NOMINAL_HBM_GBS = 8000.0


def time_metric_configs(names, replays, warmup, torch, w4, peaks, l2):
    """Median and min time per call of each named decode workload: `replays`
    CUDA-graph replays of L calls on distinct weight copies (L such that one
    replay streams >= 4x L2, so every call reads its weights from HBM)."""
    rows = []
    for name in names:
        wl = WORKLOADS[name]
        per = layer_bytes(wl.M, wl.N, wl.K, wl.g, wl.symmetric, wl.act).total
        L = copies_for(per, l2)
        layer = Layer(name, L, torch, w4)
        t = []
        time_graph(layer, replays, warmup, torch, lambda: None, per_step=t)
        t = [v / L for v in t]
        med, mn = statistics.median(t), min(t)
        rows.append({"workload": name, "M": wl.M, "N": wl.N, "K": wl.K, "g": wl.g, "dtype": wl.act,
                     "calls_per_replay": L, "replays": replays,
                     "us_median": round(med * 1e6, 3), "us_min": round(mn * 1e6, 3),
                     "GBs_median": round(per / med / 1e9, 1),
                     "frac_measured_hbm": round(per / med / 1e9 / peaks["hbm_gbs"], 4),
                     "frac_nominal_8tbs": round(per / med / 1e9 / NOMINAL_HBM_GBS, 4),
                     "algorithmic_bytes_per_call": per})
        del layer
        torch.cuda.empty_cache()
    return rows


def copies_for(bytes_per_layer, l2_bytes):
    """Enough weight copies that one step moves >= 1 GB and >= 4x L2."""
    target = max(1e9, 4 * l2_bytes)
    return int(min(128, max(4, math.ceil(target / bytes_per_layer))))


def run_ours(args, rank, world, barrier, allmax):
    import torch

    import weight_only_int4_gb300 as w4
    if not os.path.exists(w4.LIB_PATH):
        if rank == 0:
            from weight_only_int4_gb300 import build as b
            b.build()
        barrier()
    w4.load_library()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    peaks, peak_src = load_peaks()

    wl = WORKLOADS[args.workload]
    per_layer = layer_bytes(wl.M, wl.N, wl.K, wl.g, wl.symmetric, wl.act).total
    L = max(copies_for(per_layer, l2), args.layers)
    copy_gbs = box_copy_gbs(torch)
    layer = Layer(args.workload, L, torch, w4)

    clocks = ClockSampler(local)
    clocks.start()
    step_s = []
    secs = time_graph(layer, args.steps, args.warmup, torch, barrier, per_step=step_s)
    clk = clocks.stop()
    secs = allmax(secs)
    launches = args.steps * L
    ms_per_step = secs * 1e3 / args.steps
    launch_s = secs / launches
    bytes_per_launch = layer.bytes.total
    value = world * args.steps * L * bytes_per_launch / secs / 1e9
    achieved = bytes_per_launch / launch_s / 1e9

    e2e_steps = max(3, args.steps // 4)
    e2e_s, h2d, d2h = time_e2e(layer, e2e_steps, args.warmup, torch)
    e2e_s = allmax(e2e_s)
    e2e_value = world * e2e_steps * L * bytes_per_launch / e2e_s / 1e9
    if w4.device_status() != w4.OK:
        raise RuntimeError("device-side error status after the timed region")

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.act,
        "data": "synthetic (seeded: x~N(0,1), q,z~U{0..15}, s~U[0.002,0.02])",
        "config": {"workload": args.workload, "M": wl.M, "N": wl.N, "K": wl.K, "g": wl.g,
                   "layers_per_step": L, "parallelism": f"replicas x{world}",
                   "step": f"one CUDA graph of {L} GEMV calls on distinct weight copies (a decode step of "
                           f"{L} layers' gate_up projections)",
                   "l2": f"each step streams {L} distinct weight copies "
                         f"({L * per_layer / 1e6:.0f} MB > L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA-graph replay of one step, CUDA events on the replay stream"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peak_src,
                     "traffic": load_traffic("gemv", args.workload),
                     "kernel": "gemv_kernel", "algorithmic_bytes_per_launch": bytes_per_launch,
                     "us_per_launch": round(launch_s * 1e6, 3),
                     "us_per_launch_median": round(statistics.median(step_s) / L * 1e6, 3),
                     "us_per_launch_min": round(min(step_s) / L * 1e6, 3),
                     "frac_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "context": {"this_gpu_copy_gbs": copy_gbs,
                                 "frac_of_this_gpu_copy": round(achieved / copy_gbs, 4)}},
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": "pinned x -> device, L public-API gemv calls, every y -> pinned host"},
        "gpu_launches": launches,
    }
    del layer
    torch.cuda.empty_cache()

    if not args.no_configs:
        clocks = ClockSampler(local)
        clocks.start()
        rows = time_metric_configs(METRIC_CONFIGS, max(50, args.config_replays), max(3, args.warmup), torch,
                                   w4, peaks, l2)
        cclk = clocks.stop()
        line["configs"] = {"rows": rows, "clocks": cclk, "peak_source": peak_src,
                           "timing": "per-replay CUDA events around a CUDA graph of L calls on distinct "
                                     "weight copies; per call = replay / L; median and min over the replays"}
        line["gpu_launches"] += sum(r["calls_per_replay"] * r["replays"] for r in rows)

    if not args.no_prefill:
        pw = WORKLOADS[PREFILL]
        pre = Layer(PREFILL, 2, torch, w4)
        psteps = max(3, args.steps // 20)
        clocks = ClockSampler(local)
        clocks.start()
        psecs = allmax(time_graph(pre, psteps, max(3, args.warmup), torch, barrier))
        pclk = clocks.stop()
        plaunch = psecs / (psteps * 2)
        tflops = pre.flops / plaunch / 1e12
        line["prefill"] = {
            "workload": PREFILL, "M": pw.M, "N": pw.N, "K": pw.K, "g": pw.g, "dtype": pw.act,
            "value": round(world * tflops, 1), "unit": "TFLOP/s", "ms_per_call": round(plaunch * 1e3, 4),
            "calls": psteps * 2,
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tflops / peaks["bf16_tflops"], 4),
                         "peak_source": peak_src + " (burst)",
                         "traffic": load_traffic("gemm", PREFILL), "kernel": "gemm_kernel",
                         "algorithmic_flops_per_launch": pre.flops},
            "clocks": pclk,
        }
        line["gpu_launches"] += psteps * 2
        del pre
        torch.cuda.empty_cache()

    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    return line


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(name, cols):
    """Operands of the workload restricted to the first `cols` columns (same seed)."""
    from oracle import w4a16_oracle as O
    wl = WORKLOADS[name]
    case = wl.case(seed=0)
    q = np.ascontiguousarray(case.q[:, :cols])
    z = None if case.z is None else np.ascontiguousarray(case.z[:, :cols])
    s = np.ascontiguousarray(case.s[:, :cols])
    return wl, case.x, O.pack_rows(q), s, (None if z is None else O.pack_cols(z))


# Output columns of the workload in the oracle's sample; the CPU baseline of
# the default line and the reference arm time the same sample.
ORACLE_COLS = 1024


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(name, budget_s=15.0, cols=ORACLE_COLS):
    from oracle import w4a16_oracle as O
    wl, x, qw, s, qz = oracle_sample(name, cols)
    bytes_sample = layer_bytes(wl.M, cols, wl.K, wl.g, wl.symmetric, wl.act).total
    n, t_wall, t_cpu = 0, 0.0, 0.0
    while t_wall < budget_s:
        c0, w0 = time.process_time(), time.perf_counter()
        O.reference(x, qw, s, qz, wl.g, wl.act)
        t_cpu += time.process_time() - c0
        t_wall += time.perf_counter() - w0
        n += 1
    return {"value": round(n * bytes_sample / t_wall / 1e9, 4), "unit": "GB/s",
            "cores": max(1, round(t_cpu / t_wall)), "kind": "oracle",
            "sample": f"{n} x oracle on columns [0,{cols}) of {name} ({bytes_sample} B each)",
            "host_cpus": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args):
    from oracle import w4a16_oracle as O
    cols = ORACLE_COLS
    wl, x, qw, s, qz = oracle_sample(args.workload, cols)
    bytes_sample = layer_bytes(wl.M, cols, wl.K, wl.g, wl.symmetric, wl.act).total
    for _ in range(args.warmup):
        O.reference(x, qw, s, qz, wl.g, wl.act)
    c0, w0 = time.process_time(), time.perf_counter()
    for _ in range(args.steps):
        O.reference(x, qw, s, qz, wl.g, wl.act)
    wall = time.perf_counter() - w0
    cpu = time.process_time() - c0
    value = args.steps * bytes_sample / wall / 1e9
    sample = f"oracle on columns [0,{cols}) of {args.workload} per step ({bytes_sample} B)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": args.workload, "M": wl.M, "N": wl.N, "K": wl.K,
                                                  "g": wl.g},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": max(1, round(cpu / wall)),
                         "kind": "oracle", "sample": sample, "host_cpus": os.cpu_count(),
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def dist_helpers(device):
    """Barrier and max-over-ranks of a float for the replicas (the process group
    is already initialised): every rank's timed region is bracketed by the
    barrier, and the job's time is the slowest rank's."""
    import torch
    import torch.distributed as dist

    def barrier():
        dist.barrier()

    def allmax(v):
        t = torch.tensor([v], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, allmax


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DECODE, choices=[n for n, w in WORKLOADS.items() if w.kernel == "gemv"])
    ap.add_argument("--layers", type=int, default=32,
                    help="layers (distinct weight copies) per decode step, like one decode step of a 32-layer "
                         "decoder captured as one graph; at least enough to exceed 4x L2")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config rows (M = 1-4 decode workloads beside the headline)")
    ap.add_argument("--config-replays", type=int, default=60,
                    help="CUDA-graph replays per config row (at least 50)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--configs", action="store_true", help="time every named workload (one GPU) and exit")
    ap.add_argument("--match", default="", help="with --configs: only workloads whose name contains this")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.configs:
        if rank == 0:
            print(json.dumps(run_configs(args)), flush=True)
        return

    barrier = lambda: None  # noqa: E731
    allmax = lambda v: v    # noqa: E731
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
        barrier, allmax = dist_helpers("cuda")

    line = run_ours(args, rank, world, barrier, allmax)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
