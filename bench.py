#!/usr/bin/env python
"""Benchmark of the FP8 E4M3 quantized linear layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--headline-only]

One JSON line on stdout (rank 0).  A step is one pass of the layer over every
shape of the workload:
  * decode_w8a16 (default; the decode workload of the W8A16 path): the 12
    fp16 x E4M3 products M in {1,4,16} x (N,K) in {(12288,4096),
    (4096,4096), (22016,4096), (4096,11008)}; metric GB/s of algorithmic
    bytes (2MK + NK + 2MN + 4N per product).
  * prefill_w8a8_outliers / llama3_8b_w8a8_sweep / llama70b_static_fp8out:
    activation quantization (dynamic or static) plus the W8A8 product of
    every shape; metric TFLOP/s (2MNK), M <= 16 shapes also in GB/s.
Weights are quantized once before timing (untimed setup), as the layer does
after loading; W8A16 weights are then packed into the kernel's fragment
order (--w8a16-layout row-major keeps [N, K] rows).  Each shape owns its own weight buffer and, where a step's
footprint is below 3x the L2 size, the inputs rotate over several copies,
so every timed step reads its operands from HBM.

The timed region replays a CUDA graph of one step K times (after W warm-up
replays), bracketed by CUDA events on the launching stream; event-record
nodes inside the graph time each kernel call, which gives the roofline
figure of the dominant kernel.  The end-to-end figure runs the public API
eagerly with pinned host buffers: host-to-device copies of the activations,
the kernels, and device-to-host copies of the outputs, every step.

--impl reference times the CPU oracle (plain C loops, one thread) on a
bounded sample of the same workload, in the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

METRIC = "FP8 scaled-GEMM TFLOP/s (GB/s at M<=16) and % of GB300 roofline"
L2_BYTES = 126 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor rate ratio (4.5 / 2.25 PFLOP/s)


# ----------------------------------------------------------------------------- utilities

def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode_w8a16", choices=sorted(synthetic.WORKLOADS))
    p.add_argument("--headline-only", action="store_true",
                   help="skip the other workloads' summary entries")
    p.add_argument("--extra-steps", type=int, default=20)
    p.add_argument("--w8a16-layout", choices=["packed", "row-major"], default="packed",
                   help="weights of the W8A16 products: packed once at setup into the "
                        "kernel's fragment order (fp8_pack_w8a16_weights), or [N, K] rows")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.steps < 1:
        p.error("--steps must be >= 1")
    return args


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_step: float, ms_per_step: float, world: int, unit: str) -> float:
    """Whole-job throughput of N replicas: every rank processes the same
    units per step; the step time is the maximum over ranks."""
    sec = ms_per_step / 1e3
    scale = 1e9 if unit == "GB/s" else 1e12
    return units_per_step * world / sec / scale


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 25 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.samples = []
        self.proc = None
        self.thread = None
        self.gpu = self._gpu_id(device)

    @staticmethod
    def _gpu_id(device):
        props = torch.cuda.get_device_properties(device)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", 0)
        devid = getattr(props, "pci_device_id", 0)
        if bus is None:
            return None
        return f"{dom:08X}:{bus:02X}:{devid:02X}.0"

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "25"]
        if self.gpu:
            cmd += ["-i", self.gpu]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.2)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append((time.perf_counter(), float(parts[1]), float(parts[2]),
                                     float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                                     parts[5:9]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1, tw0):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if len(inside) < 3:
            inside = [s for s in self.samples if tw0 <= s[0] <= t1]
            window = "warmup+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": window}
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[4])
                          if v.lower() == "active"})
        return {"sm_mhz": float(np.median([s[1] for s in inside])),
                "sm_max_mhz": float(max(s[2] for s in inside)),
                "power_w_max": float(max(s[3] for s in inside)),
                "reasons": reasons, "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------- workloads

def w8a16_bytes(M, N, K):
    return 2 * M * K + N * K + 2 * M * N + 4 * N


def w8a8_bytes(M, N, K, out_bytes, per_channel):
    return M * K + N * K + M * N * out_bytes + 4 * (N if per_channel else 1) + 4


class Call:
    """One public-API call inside a step (1 or 2 kernel launches)."""

    def __init__(self, kind, fn, units, unit, launches, shape):
        self.kind, self.fn, self.units, self.unit = kind, fn, units, unit
        self.launches, self.shape = launches, shape


class Workload:
    def __init__(self, name, device, packed_w8a16=True):
        import fp8_quantized_linear_gb300 as fl
        self.fl = fl
        self.name = name
        self.packed = packed_w8a16 and synthetic.WORKLOADS[name].kind == "w8a16"
        self.wl = synthetic.WORKLOADS[name]
        self.device = device
        self.copies = []      # per rotation copy: list of per-shape dicts
        self.rot = 1

    # -- setup --
    def build(self):
        wl, dev, fl = self.wl, self.device, self.fl
        host = []
        for i, (M, N, K) in enumerate(wl.shapes):
            seed = wl.seed(i)
            x = synthetic.activation(M, K, wl.x_dtype, seed=seed, outlier_frac=wl.outlier_frac)
            host.append((M, N, K, seed, x))
        # one copy first, then decide the rotation count from its footprint
        first, foot = self._make_copy(host, weights_cache={})
        self.copies.append(first)
        self.rot = max(1, min(16, math.ceil(3 * L2_BYTES / max(foot, 1))))
        for _ in range(self.rot - 1):
            self.copies.append(self._clone_copy(first))
        self.footprint = foot
        torch.cuda.synchronize(dev)

    def _make_copy(self, host, weights_cache):
        wl, dev, fl = self.wl, self.device, self.fl
        items, foot = [], 0
        for (M, N, K, seed, x) in host:
            key = (N, K)
            if key not in weights_cache:
                weights_cache[key] = synthetic.weight(N, K, torch.bfloat16, seed=seed).to(dev)
            wbf = weights_cache[key]
            it = {"M": M, "N": N, "K": K, "x": x.to(dev)}
            if wl.kind == "w8a16":
                it["qw"], it["sw"] = fl.fp8_quant_per_row(wbf)
                if self.packed:
                    it["qw"] = fl.fp8_pack_w8a16_weights(it["qw"])
                it["y"] = torch.empty((M, N), dtype=wl.x_dtype, device=dev)
                foot += w8a16_bytes(M, N, K)
            else:
                if wl.w_scale == "channel":
                    it["qw"], it["sw"] = fl.fp8_quant_per_row(wbf)
                else:
                    it["qw"], it["sw"] = fl.fp8_quant_per_tensor(wbf)
                it["qa"] = torch.empty((M, K), dtype=torch.uint8, device=dev)
                it["sa"] = torch.empty(1, dtype=torch.float32, device=dev)
                if wl.act_scale == "static":
                    calib = synthetic.activation(256, K, wl.x_dtype,
                                                 seed=synthetic.calibration_seed(seed)).to(dev)
                    _, sa = fl.fp8_quant_per_tensor(calib)
                    it["sa"].copy_(sa)
                    qc, _ = fl.fp8_quant_per_tensor(calib, scale=sa, dynamic=False)
                    yc = fl.fp8_scaled_mm(qc, it["qw"], sa, it["sw"], out_dtype=torch.float16)
                    # output_scale = amax of the calibration output / 448: the
                    # library's dynamic scale of that output gives exactly this
                    _, it["os"] = fl.fp8_quant_per_tensor(yc)
                out_dt = {"bf16": torch.bfloat16, "fp16": torch.float16,
                          "e4m3": torch.uint8}[wl.out_dtype]
                it["y"] = torch.empty((M, N), dtype=out_dt, device=dev)
                foot += w8a8_bytes(M, N, K, it["y"].element_size(), wl.w_scale == "channel")
                foot += 2 * M * K  # activation read by the quantizer
            items.append(it)
        weights_cache.clear()
        return items, foot

    def _clone_copy(self, items):
        out = []
        for it in items:
            out.append({k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in it.items()})
        return out

    # -- one step's calls on copy r --
    def calls(self, r):
        fl, wl = self.fl, self.wl
        ws = fl.workspace(self.device)
        out = []
        for it in self.copies[r]:
            M, N, K = it["M"], it["N"], it["K"]
            if wl.kind == "w8a16":
                out.append(Call("w8a16_skinny",
                                lambda it=it: fl.fp8_w8a16_mm(it["x"], it["qw"], it["sw"], y=it["y"],
                                                              stable_weights=True,
                                                              packed=self.packed),
                                w8a16_bytes(M, N, K), "bytes", 1, (M, N, K)))
                continue
            dynamic = wl.act_scale == "dynamic"
            out.append(Call("quant_dynamic" if dynamic else "quant_static",
                            lambda it=it, dyn=dynamic: fl.fp8_quant_per_tensor(
                                it["x"], q=it["qa"], scale=it["sa"], dynamic=dyn, ws=ws),
                            3 * M * K, "bytes", 1, (M, N, K)))
            kind = "scaled_mm_skinny" if M <= 16 else "scaled_mm_tcgen05"
            units = (w8a8_bytes(M, N, K, it["y"].element_size(), wl.w_scale == "channel")
                     if M <= 16 else 2 * M * N * K)
            out.append(Call(kind,
                            lambda it=it: fl.fp8_scaled_mm(it["qa"], it["qw"], it["sa"], it["sw"],
                                                           out_dtype=it["y"].dtype,
                                                           out_scale=it.get("os"), y=it["y"],
                                                           ws=ws, stable_weights=True),
                            units, "bytes" if M <= 16 else "flops", 1, (M, N, K)))
        return out

    def step_units(self):
        """(bytes, flops) of one step: the workload's headline quantity."""
        b = f = 0
        for it in self.copies[0]:
            M, N, K = it["M"], it["N"], it["K"]
            if self.wl.kind == "w8a16":
                b += w8a16_bytes(M, N, K)
            else:
                b += w8a8_bytes(M, N, K, it["y"].element_size(), self.wl.w_scale == "channel")
            f += 2 * M * N * K
        return b, f

    def headline_unit(self):
        return "GB/s" if self.wl.kind == "w8a16" else "TFLOP/s"

    # -- end to end through the public API with host buffers --
    def e2e(self, steps):
        """Seconds per step of the whole workload from host memory to host
        memory: one pinned host -> device copy of all the step's activations,
        the public-API call(s) of every product, and one device -> pinned host
        copy of all its outputs.  Measured twice: with the step's calls and copies captured
        in one CUDA graph replayed once per step (how a serving loop runs a
        fixed step), and with the same calls issued eagerly.  Every step ends
        with a host synchronize.  Returns (graph s, eager s, h2d bytes, d2h
        bytes)."""
        fl, wl, dev = self.fl, self.wl, self.device
        items = self.copies[0]
        # the step's activations in one pinned host buffer and one device
        # buffer (each product's block starts on a 256-byte boundary), the
        # outputs likewise: one copy each way per step
        def packed(tensors):
            offs, total = [], 0
            for t in tensors:
                offs.append(total)
                total += (t.numel() * t.element_size() + 255) // 256 * 256
            return offs, total
        x_offs, x_total = packed([it["x"] for it in items])
        y_offs, y_total = packed([it["y"] for it in items])
        x_host = torch.empty(x_total, dtype=torch.uint8).pin_memory()
        y_host = torch.empty(y_total, dtype=torch.uint8).pin_memory()
        x_dev = torch.empty(x_total, dtype=torch.uint8, device=dev)
        y_dev = torch.empty(y_total, dtype=torch.uint8, device=dev)
        xs, ys = [], []
        for it, xo, yo in zip(items, x_offs, y_offs):
            nx = it["x"].numel() * it["x"].element_size()
            ny = it["y"].numel() * it["y"].element_size()
            x_host[xo:xo + nx].copy_(it["x"].reshape(-1).view(torch.uint8).cpu())
            xs.append(x_dev[xo:xo + nx].view(it["x"].dtype).view(it["x"].shape))
            ys.append(y_dev[yo:yo + ny].view(it["y"].dtype).view(it["y"].shape))
        h2d, d2h = x_total, y_total
        ws = fl.workspace(dev)

        def body():
            x_dev.copy_(x_host, non_blocking=True)
            for it, x, y in zip(items, xs, ys):
                if wl.kind == "w8a16":
                    fl.fp8_w8a16_mm(x, it["qw"], it["sw"], y=y, stable_weights=True,
                                    packed=self.packed)
                else:
                    fl.fp8_quant_per_tensor(x, q=it["qa"], scale=it["sa"],
                                            dynamic=wl.act_scale == "dynamic", ws=ws)
                    fl.fp8_scaled_mm(it["qa"], it["qw"], it["sa"], it["sw"],
                                     out_dtype=y.dtype, out_scale=it.get("os"),
                                     y=y, ws=ws, stable_weights=True)
            y_host.copy_(y_dev, non_blocking=True)

        stream = torch.cuda.Stream(dev)
        with torch.cuda.stream(stream):
            for _ in range(3):
                body()
                stream.synchronize()
            t0 = time.perf_counter()
            for _ in range(steps):
                body()
                stream.synchronize()
            eager = (time.perf_counter() - t0) / steps
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
                stream.synchronize()
            t0 = time.perf_counter()
            for _ in range(steps):
                g.replay()
                stream.synchronize()
            graph = (time.perf_counter() - t0) / steps
        return graph, eager, h2d, d2h

    # -- CPU oracle on a bounded sample --
    def prepare_cpu_sample(self, fraction=1.0):
        """Oracle inputs for a sample of this workload: (jobs, units of the
        headline metric, description).  W8A16: the first fraction*N output
        channels of every product (per-row scales are row-local, so these are
        exactly the workload's values).  W8A8: 8 activation rows and the
        first 1024*fraction weight rows of every shape (a timing sample)."""
        import oracle
        wl = self.wl
        oracle.build()
        jobs, units = [], 0
        if wl.kind == "w8a16":
            for i, (M, N, K) in enumerate(wl.shapes):
                seed = wl.seed(i)
                n_s = min(N, max(16, int(N * fraction) // 16 * 16))
                x = synthetic.activation(M, K, wl.x_dtype, seed=seed)
                w = synthetic.weight(N, K, torch.bfloat16, seed=seed, row_subset=range(n_s))
                qw, sw = oracle.quant_per_row(w)
                jobs.append(("w8a16", x, qw, sw))
                units += w8a16_bytes(M, n_s, K)
            desc = (f"first {fraction:.0%} of the output channels of all 12 products "
                    f"(brute-force C loops, 1 thread)")
            return jobs, units, desc
        rows = 8
        for i, (M, N, K) in enumerate(wl.shapes):
            seed = wl.seed(i)
            r = min(rows, M)
            n_s = min(N, max(16, int(1024 * fraction) // 16 * 16))
            x = synthetic.activation(M, K, wl.x_dtype, seed=seed, outlier_frac=wl.outlier_frac,
                                     row_subset=list(range(r)))
            w = synthetic.weight(N, K, torch.bfloat16, seed=seed, row_subset=range(n_s))
            if wl.w_scale == "channel":
                qw, sw = oracle.quant_per_row(w)
            else:
                qw, s = oracle.quant_per_tensor(w)
                sw = np.array([s], np.float32)
            jobs.append(("w8a8", x, qw, sw))
            units += 2 * r * n_s * K
        desc = (f"{rows} activation rows x the first {n_s} weight rows of every shape: "
                f"quantize + brute-force C product, 1 thread")
        return jobs, units, desc

    @staticmethod
    def run_cpu_sample(jobs):
        import oracle
        t0 = time.perf_counter()
        for kind, x, qw, sw in jobs:
            if kind == "w8a16":
                oracle.w8a16_bruteforce(x, qw, sw)
            else:
                qa, sa = oracle.quant_per_tensor(x)
                oracle.scaled_mm_bruteforce(qa, qw, sa, sw)
        return time.perf_counter() - t0


# ----------------------------------------------------------------------------- measurement

def _event(external):
    if external:
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None
    return torch.cuda.Event(enable_timing=True)


def measure(work: Workload, steps: int, warmup: int, world: int, sampler=None):
    """Times `steps` replays of a CUDA graph of one step (no instrumentation
    inside it), then replays a second graph of the same step with an event
    node around every call to split the step time among the kernels."""
    dev = work.device
    stream = torch.cuda.Stream(device=dev)
    # eager pass: initializes the library (device check, shared-memory
    # attribute, TMA encoder) and the workspace outside any capture
    with torch.cuda.stream(stream):
        for r in range(work.rot):
            for c in work.calls(r):
                c.fn()
    stream.synchronize()
    graphs, inst, evsets, call_lists = [], [], [], []
    have_external = _event(True) is not None
    for r in range(work.rot):
        calls = work.calls(r)
        call_lists.append(calls)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c.fn()
        graphs.append(g)
        if have_external:
            evs = [_event(True) for _ in range(len(calls) + 1)]
            gi = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gi, stream=stream):
                for i, c in enumerate(calls):
                    evs[i].record()
                    c.fn()
                evs[-1].record()
            inst.append(gi)
            evsets.append(evs)
    torch.cuda.synchronize(dev)

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        tw0 = time.perf_counter()
        for s in range(warmup):
            graphs[s % work.rot].replay()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        start.record(stream)
        for s in range(steps):
            graphs[s % work.rot].replay()
        stop.record(stream)
        stop.synchronize()
        t1 = time.perf_counter()
        barrier(world)
        torch.cuda.synchronize(dev)
    ms_total = start.elapsed_time(stop)
    ms_total = reduce_max(ms_total, world, dev)

    # per-call shares from the instrumented graphs (after the timed region)
    per_kind = {}
    if have_external:
        reps = max(3, min(20, steps))
        with torch.cuda.stream(stream):
            for rep in range(reps):
                r = rep % work.rot
                inst[r].replay()
                stream.synchronize()
                evs = evsets[r]
                for i, c in enumerate(call_lists[r]):
                    d = evs[i].elapsed_time(evs[i + 1])
                    k = per_kind.setdefault(c.kind, {"ms": 0.0, "units": 0, "unit": c.unit,
                                                     "calls": 0, "launches": 0})
                    k["ms"] += d
                    k["units"] += c.units
                    k["calls"] += 1
                    k["launches"] += c.launches
        for k in per_kind.values():
            k["units_per_step"] = k["units"] / reps
            k["launches_per_step"] = k["launches"] / reps
    launches_per_step = sum(c.launches for c in call_lists[0])
    return {"ms_total": ms_total, "ms_per_step": ms_total / steps, "per_kind": per_kind,
            "kernel_timing": ("shares from event nodes in a separate replay of the step graph; "
                              "kernel time = timed step time x share") if have_external else "none",
            "gpu_launches": launches_per_step * steps, "window": (tw0, t0, t1)}


def roofline(per_kind, peaks, ms_per_step):
    """Roofline of the dominant kernel: its algorithmic units per step over
    its time per step (the timed step time times its measured share)."""
    if not per_kind:
        return None, None
    total = sum(v["ms"] for v in per_kind.values())
    kind, v = max(per_kind.items(), key=lambda kv: kv[1]["ms"])
    share = v["ms"] / total if total > 0 else 1.0
    secs = ms_per_step * share / 1e3
    ups = v["units_per_step"]
    if v["unit"] == "flops":
        achieved = ups / secs / 1e12
        peak = peaks["bf16_tflops"] * FP8_OVER_BF16
        rf = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
              "unit": "TFLOP/s", "frac": round(achieved / peak, 4)}
        rf["peak_source"] = (f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} TFLOP/s x "
                             f"{FP8_OVER_BF16} (nominal FP8/BF16 dense ratio)")
    else:
        achieved = ups / secs / 1e9
        peak = peaks["hbm_gbs"]
        rf = {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(peak, 1),
              "unit": "GB/s", "frac": round(achieved / peak, 4)}
        rf["peak_source"] = f"{peaks['source']} HBM copy bandwidth"
    rf["kernel"] = kind
    rf["share"] = round(share, 4)
    rf["launches_per_step"] = v["launches_per_step"]
    rf["traffic"] = traffic_from_profile(kind)
    return rf, {k: {"share": round(x["ms"] / total, 4) if total else None,
                    "launches_per_step": x["launches_per_step"]} for k, x in per_kind.items()}


KERNEL_SOURCES = {"w8a16_skinny": "skinny.cu", "scaled_mm_skinny": "skinny.cu",
                  "scaled_mm_tcgen05": "gemm_tcgen05.cu", "quant_dynamic": "quant.cu",
                  "quant_static": "quant.cu"}


def kernel_source_hash(src):
    """sha256 prefix of a kernel's translation unit followed by the shared
    header it includes (a change to either invalidates a capture)."""
    csrc = os.path.join(ROOT, "fp8_quantized_linear_gb300", "csrc")
    h = hashlib.sha256()
    for name in (src, "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kind):
    """DRAM bytes of one captured launch of this kernel, from the committed ncu
    summary, if the kernel source still has the hash the capture was taken
    with (else None).  Returns {"bytes", "algorithmic_bytes", "launch"}."""
    src = KERNEL_SOURCES.get(kind)
    if src is None:
        return None
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    h = kernel_source_hash(src)
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) == 5 and cells[0] == kind and cells[1] == h:
            return {"bytes": int(cells[2]), "algorithmic_bytes": int(cells[3]),
                    "launch": cells[4]}
    return None


# ----------------------------------------------------------------------------- arms

def run_ours(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    work = Workload(args.workload, dev, packed_w8a16=args.w8a16_layout == "packed")
    work.build()
    sampler = ClockSampler(dev)
    sampler.start()
    res = measure(work, args.steps, args.warmup, world)
    sampler.stop()
    clocks = sampler.summary(res["window"][1], res["window"][2], res["window"][0])
    b, f = work.step_units()
    unit = work.headline_unit()
    value = aggregate(b if unit == "GB/s" else f, res["ms_per_step"], world, unit)
    rf, kinds = roofline(res["per_kind"], peaks, res["ms_per_step"])
    # end to end through the public API with host buffers
    e2e_steps = max(3, min(args.steps, 50))
    dt_e2e, dt_eager, h2d, d2h = work.e2e(e2e_steps)
    e2e_val = ((b / dt_e2e / 1e9) if unit == "GB/s" else (f / dt_e2e / 1e12)) * world
    e2e_eager = ((b / dt_eager / 1e9) if unit == "GB/s" else (f / dt_eager / 1e12)) * world
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(res["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 x e4m3 (fp32 accumulate)" if work.wl.kind == "w8a16"
                 else "e4m3 x e4m3 (fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": work.name, "description": work.wl.description,
                   "shapes": [list(s) for s in work.wl.shapes],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": (f"inputs larger than L2: {work.footprint / 2**20:.0f} MiB per step"
                          + (f" x {work.rot} rotating copies" if work.rot > 1 else "")),
                   "graph": "one CUDA graph per step",
                   **({"weights": ("E4M3 codes packed once at setup into the kernel's fragment "
                                   "order (fp8_pack_w8a16_weights)" if work.packed
                                   else "E4M3 codes as [N, K] rows")}
                      if work.wl.kind == "w8a16" else {})},
        "roofline": rf, "kernels": kinds, "kernel_timing": res["kernel_timing"],
        "e2e": {"value": round(e2e_val, 3), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "api": "one pinned host->device copy of the step's activations, the "
                       "fp8_quantized_linear_gb300 calls, one device->pinned host copy of the "
                       "outputs, captured in one CUDA graph, replayed and synchronized once "
                       "per step",
                "eager_value": round(e2e_eager, 3),
                "eager_api": "the same calls and copies issued eagerly, synchronized per step"},
        "gpu_launches": res["gpu_launches"], "clocks": clocks,
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "source")},
    }
    if rank == 0:
        jobs, units, desc = work.prepare_cpu_sample(1.0)
        secs = Workload.run_cpu_sample(jobs)
        cpu_val = (units / secs / 1e9) if unit == "GB/s" else (units / secs / 1e12)
        line["cpu_baseline"] = {"value": round(cpu_val, 6), "unit": unit, "cores": 1,
                                "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
        if not args.headline_only and work.name == "decode_w8a16":
            line["workloads"] = other_workloads(args, dev, peaks)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def other_workloads(args, dev, peaks):
    """Short measurements of the W8A8 workloads (summary entries)."""
    out = []
    for name in ("prefill_w8a8_outliers", "llama3_8b_w8a8_sweep", "llama70b_static_fp8out"):
        work = Workload(name, dev)
        work.build()
        res = measure(work, args.extra_steps, max(3, args.warmup // 2), 1)
        b, f = work.step_units()
        sec = res["ms_per_step"] / 1e3
        rf, kinds = roofline(res["per_kind"], peaks, res["ms_per_step"])
        entry = {"workload": name, "value": round(f / sec / 1e12, 2), "unit": "TFLOP/s",
                 "ms_per_step": round(res["ms_per_step"], 4), "steps": args.extra_steps,
                 "roofline": rf, "kernels": kinds}
        entry["per_shape"] = per_shape(work, args.extra_steps)
        out.append(entry)
        del work
        torch.cuda.empty_cache()
    return out


def per_shape(work, steps):
    """Per-shape product times: eager calls bracketed by events, L2 flushed
    before each timed call (the activation quantization of W8A8 shapes runs
    untimed just before its product)."""
    rows = []
    calls_by_copy = [work.calls(r) for r in range(work.rot)]
    per = 1 if work.wl.kind == "w8a16" else 2
    stream = torch.cuda.current_stream(work.device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=work.device)
    reps = max(3, steps // 2)
    for j in range(len(work.wl.shapes)):
        tot_ms = 0.0
        for rep in range(reps):
            cc = calls_by_copy[rep % work.rot]
            flush.zero_()
            if per == 2:
                cc[2 * j].fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            cc[per * j + per - 1].fn()
            b.record(stream)
            b.synchronize()
            tot_ms += a.elapsed_time(b)
        c = calls_by_copy[0][per * j + per - 1]
        M, N, K = c.shape
        ms = tot_ms / reps
        row = {"M": M, "N": N, "K": K, "kernel": c.kind, "us": round(ms * 1e3, 2),
               "TFLOP/s": round(2 * M * N * K / (ms / 1e3) / 1e12, 2)}
        if c.unit == "bytes":
            row["GB/s"] = round(c.units / (ms / 1e3) / 1e9, 1)
        rows.append(row)
    del flush
    return rows


def run_reference(args):
    """The CPU oracle, as it stands, timed on this host on a bounded sample of
    the workload: each step runs the same sample, sized so that warm-up plus
    timed steps take about two minutes."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    wl = synthetic.WORKLOADS[args.workload]
    work = Workload.__new__(Workload)
    work.wl, work.name = wl, args.workload
    unit = "GB/s" if wl.kind == "w8a16" else "TFLOP/s"
    probe_jobs, _, _ = work.prepare_cpu_sample(1.0 / 16)
    t_probe = Workload.run_cpu_sample(probe_jobs) * 16
    fraction = min(1.0, 120.0 / max(t_probe * (args.steps + args.warmup), 1e-9))
    jobs, units, desc = work.prepare_cpu_sample(fraction)
    for _ in range(args.warmup):
        Workload.run_cpu_sample(jobs)
    tot_t = 0.0
    for _ in range(args.steps):
        tot_t += Workload.run_cpu_sample(jobs)
    val = (units * args.steps / tot_t / 1e9) if unit == "GB/s" else (units * args.steps / tot_t / 1e12)
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot_t / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "description": wl.description,
                       "shapes": [list(sh) for sh in wl.shapes],
                       "parallelism": "rank 0 only (host cores)"},
            "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": desc, "value": round(val, 6),
                             "unit": unit},
            "e2e": {"value": round(val, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
