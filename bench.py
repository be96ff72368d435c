#!/usr/bin/env python
"""Benchmark of the FP8 E4M3 quantized linear layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--headline-only]

One JSON line on stdout (rank 0).  A step is one pass of the layer over every
shape of the workload:
  * llama70b_static_fp8out (default, the largest workload): static
    activation quantization plus the W8A8 product with per-channel weight
    scales and E4M3 output (output_scale) of 16 shapes, M in {1,64,1024,4096}
    x (N,K) in {(10240,8192),(8192,8192),(57344,8192),(8192,28672)}; metric
    TFLOP/s (2MNK).
  * decode_w8a16: the 12 fp16 x E4M3 products M in {1,4,16} x (N,K) in
    {(12288,4096), (4096,4096), (22016,4096), (4096,11008)}; metric GB/s of
    algorithmic bytes (2MK + NK + 2MN + 4N per product).
  * prefill_w8a8_outliers / llama3_8b_w8a8_sweep / tiny_w8a8: dynamic
    activation quantization plus the W8A8 product of every shape; TFLOP/s.
With the default workload the line also carries one entry per other
workload (same measurement, shorter), and every line carries per-shape
figures: each product timed alone (a CUDA graph of the one call over
rotating operand copies, replayed back to back, CUDA events outside the
replays) against the roofline min(tensor peak, HBM bandwidth x arithmetic
intensity), and, for M <= 16, against HBM bandwidth alone.
Weights are quantized once before timing (untimed setup), as the layer does
after loading; W8A16 weights are then packed into the kernel's fragment
order (--w8a16-layout row-major keeps [N, K] rows).  Each shape owns its own weight buffer and, where a step's
footprint is below 3x the L2 size, the inputs rotate over several copies,
so every timed step reads its operands from HBM.

The timed region replays a CUDA graph of one step K times (after W warm-up
replays), bracketed by CUDA events on the launching stream; event-record
nodes inside the graph time each kernel call, which gives the roofline
figure of the dominant kernel.  The end-to-end figure runs the public API
with pinned host buffers: host-to-device copies of the activations, the
kernels, and device-to-host copies of the outputs, every step.  Clocks,
power and clock-event reasons are sampled through NVML (read-only queries)
every 2 ms during the timed region.

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
HEADLINE = "llama70b_static_fp8out"
ENTRY_WORKLOADS = ("decode_w8a16", "prefill_w8a8_outliers", "llama3_8b_w8a8_sweep", "tiny_w8a8")
HBM_TARGET = 0.70  # fraction of HBM bandwidth the M <= 16 shapes aim for
# bench names of the three W8A8 kernels fp8_scaled_mm may run
W8A8_KINDS = {"stream": "scaled_mm_skinny", "swapped": "scaled_mm_swapped",
              "tiled": "scaled_mm_tcgen05"}
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
    p.add_argument("--workload", default=HEADLINE, choices=sorted(synthetic.WORKLOADS))
    p.add_argument("--headline-only", action="store_true",
                   help="skip the other workloads' summary entries")
    p.add_argument("--extra-steps", type=int, default=20)
    p.add_argument("--only-shape", type=int, default=None,
                   help="profiling: run only this shape (index in the workload's list)")
    p.add_argument("--single-sm-tiles", action="store_true",
                   help="tuning: tensor-core products on one SM per tile (FP8L_SINGLE_SM_TILES)")
    p.add_argument("--entries", default="workloads,norm_fusion,decode_block",
                   help="entries added to the default workload's line (comma list)")
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
    """SM clock, power and clock-event reasons of the benchmark's GPU,
    sampled during the timed region.  NVML (libnvidia-ml, read-only queries)
    every 2 ms; without NVML, nvidia-smi every 25 ms."""
    NAMES = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
             0x4: "sw_power_cap"}
    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device, period=0.002):
        self.samples = []  # (time, sm_mhz, sm_max_mhz, power_w, [reason names])
        self.period = period
        self.source = None
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.bus = self._bus_id(device)

    @staticmethod
    def _bus_id(device):
        props = torch.cuda.get_device_properties(device)
        bus = getattr(props, "pci_bus_id", None)
        if bus is None:
            return None
        dom = getattr(props, "pci_domain_id", 0)
        devid = getattr(props, "pci_device_id", 0)
        return f"{dom:08X}:{bus:02X}:{devid:02X}.0"

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0 or self.bus is None:
            return None
        handle = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(self.bus.encode(), ctypes.byref(handle)) != 0:
            return None
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        u, ull = ctypes.c_uint, ctypes.c_ulonglong

        def sample():
            sm, mx, pw, rs = u(), u(), u(), ull()
            if (lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(sm)) != 0 or
                    lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) != 0):
                return None
            power = pw.value / 1e3 if lib.nvmlDeviceGetPowerUsage(handle, ctypes.byref(pw)) == 0 else 0.0
            names = ([n for bit, n in self.NAMES.items() if rs.value & bit]
                     if reasons_fn(handle, ctypes.byref(rs)) == 0 else [])
            return (time.perf_counter(), float(sm.value), float(mx.value), power, names)
        return sample if sample() is not None else None

    def start(self):
        try:
            sample = self._nvml()
        except (OSError, AttributeError):
            sample = None
        if sample is not None:
            self.source = f"nvml every {self.period * 1e3:.0f} ms"

            def loop():
                while not self.stop_flag.is_set():
                    r = sample()
                    if r is not None:
                        self.samples.append(r)
                    time.sleep(self.period)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return
        cmd = ["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "25"]
        if self.bus:
            cmd += ["-i", self.bus]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.source = "nvidia-smi every 25 ms"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def read():
            for line in self.proc.stdout:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    self.samples.append((time.perf_counter(), float(parts[1]), float(parts[2]),
                                         float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                                         [n for n, v in zip(names, parts[5:9])
                                          if v.lower() == "active"]))
                except ValueError:
                    continue
        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()
        time.sleep(0.2)

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source, "window": "timed"}
        return {"sm_mhz": float(np.median([s[1] for s in inside])),
                "sm_max_mhz": float(max(s[2] for s in inside)),
                "power_w_max": round(float(max(s[3] for s in inside)), 1),
                "reasons": sorted({n for s in inside for n in s[4]}),
                "samples": len(inside), "source": self.source, "window": "timed"}


# ----------------------------------------------------------------------------- workloads

def w8a16_bytes(M, N, K):
    return 2 * M * K + N * K + 2 * M * N + 4 * N


def w8a8_bytes(M, N, K, out_bytes, per_channel):
    return M * K + N * K + M * N * out_bytes + 4 * (N if per_channel else 1) + 4


def johnson_order(first, second):
    """Job order of Johnson's rule for a two-machine flow shop (Johnson,
    1954), which minimizes the makespan when every job runs on machine 1
    for first[i] and then on machine 2 for second[i]: the jobs with
    first <= second, by first ascending, then the others by second
    descending.  Here the machines are the host link's two directions and
    the jobs the products' input and output copies."""
    n = len(first)
    return (sorted([i for i in range(n) if first[i] <= second[i]], key=lambda i: first[i]) +
            sorted([i for i in range(n) if first[i] > second[i]], key=lambda i: -second[i]))


def fused_bytes(M, N, K, out_bytes, per_channel):
    """Algorithmic bytes of fp8_quant_scaled_mm: the 16-bit activations,
    the weights, the output and the scales."""
    return w8a8_bytes(M, N, K, out_bytes, per_channel) + M * K


class Call:
    """One public-API call inside a step (1 or 2 kernel launches)."""

    def __init__(self, kind, fn, units, unit, launches, shape):
        self.kind, self.fn, self.units, self.unit = kind, fn, units, unit
        self.launches, self.shape = launches, shape


class Workload:
    single_sm = False  # FP8L_SINGLE_SM_TILES on every product (tuning)

    def __init__(self, name, device, packed_w8a16=True, only_shape=None):
        import fp8_quantized_linear_gb300 as fl
        self.fl = fl
        self.name = name
        self.packed = packed_w8a16 and synthetic.WORKLOADS[name].kind == "w8a16"
        self.wl = synthetic.WORKLOADS[name]
        self.device = device
        self.copies = []      # per rotation copy: list of per-shape dicts
        self.rot = 1
        self.shape_ids = (list(range(len(self.wl.shapes))) if only_shape is None
                          else [only_shape])

    def shapes(self):
        """(index in the workload, (M, N, K)) of the shapes this run uses."""
        return [(i, self.wl.shapes[i]) for i in self.shape_ids]

    # -- setup --
    def build(self):
        wl, dev, fl = self.wl, self.device, self.fl
        host = []
        for i, (M, N, K) in self.shapes():
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
            if fl.quant_scaled_mm_preferred(M, N, K, dynamic):
                # quantization inside the product: 16-bit x read instead of the
                # codes; in the CUDA-core weight stream for small weights
                fused_kind = ("scaled_mm_fused_stream" if fl.scaled_mm_kernel(M, N, K) == "stream"
                              else "scaled_mm_fused_quant")
                out.append(Call(fused_kind,
                                lambda it=it, dyn=dynamic: fl.fp8_quant_scaled_mm(
                                    it["x"], it["qw"], it["sw"], a_scale=it["sa"], dynamic=dyn,
                                    out_scale=it.get("os"), y=it["y"], ws=ws, stable_weights=True),
                                fused_bytes(M, N, K, it["y"].element_size(), wl.w_scale == "channel"),
                                "bytes", 1, (M, N, K)))
                continue
            out.append(Call("quant_dynamic" if dynamic else "quant_static",
                            lambda it=it, dyn=dynamic: fl.fp8_quant_per_tensor(
                                it["x"], q=it["qa"], scale=it["sa"], dynamic=dyn, ws=ws),
                            3 * M * K, "bytes", 1, (M, N, K)))
            kind = W8A8_KINDS[fl.scaled_mm_kernel(M, N, K)]
            streams = kind != "scaled_mm_tcgen05"  # bound by reading the weights
            units = (w8a8_bytes(M, N, K, it["y"].element_size(), wl.w_scale == "channel")
                     if streams else 2 * M * N * K)
            out.append(Call(kind,
                            lambda it=it: fl.fp8_scaled_mm(it["qa"], it["qw"], it["sa"], it["sw"],
                                                           out_dtype=it["y"].dtype,
                                                           out_scale=it.get("os"), y=it["y"],
                                                           ws=ws, stable_weights=True,
                                                           single_sm=Workload.single_sm),
                            units, "bytes" if streams else "flops", 1, (M, N, K)))
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
        memory: every product's activations copied from pinned host memory,
        the public-API call(s) of every product, every output copied back to
        pinned host memory; every step ends with a host synchronize.
        Pipelined (the reported value): product i's input copy on one copy
        stream, its calls on the compute stream after that copy (an event),
        its output copy on a second copy stream after its calls, so inputs of
        later products and outputs of earlier ones cross the host link while
        the GPU computes; products in the order Johnson's rule gives for
        their input and output copies.  Serial: one copy of all activations, all calls,
        one copy of all outputs, in one stream.  Both captured in one CUDA
        graph replayed once per step (how a serving loop runs a fixed step);
        the pipelined form also issued eagerly.  Each form is timed in three
        interleaved rounds of steps/3 steps and the median round counts (the
        host link and host memory are shared with the machine's other work).
        Returns (pipelined graph s, serial graph s, pipelined eager s, h2d
        bytes, d2h bytes)."""
        fl, wl, dev = self.fl, self.wl, self.device
        items = self.copies[0]
        # the step's activations in one pinned host buffer and one device
        # buffer (each product's block starts on a 256-byte boundary), the
        # outputs likewise
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
        xs, ys, xh, xd, yh, yd = [], [], [], [], [], []
        for it, xo, yo in zip(items, x_offs, y_offs):
            nx = it["x"].numel() * it["x"].element_size()
            ny = it["y"].numel() * it["y"].element_size()
            x_host[xo:xo + nx].copy_(it["x"].reshape(-1).view(torch.uint8).cpu())
            xs.append(x_dev[xo:xo + nx].view(it["x"].dtype).view(it["x"].shape))
            ys.append(y_dev[yo:yo + ny].view(it["y"].dtype).view(it["y"].shape))
            xh.append(x_host[xo:xo + nx])
            xd.append(x_dev[xo:xo + nx])
            yh.append(y_host[yo:yo + ny])
            yd.append(y_dev[yo:yo + ny])
        h2d, d2h = x_total, y_total
        ws = fl.workspace(dev)
        dynamic = wl.act_scale == "dynamic"

        def product(it, x, y):
            if wl.kind == "w8a16":
                fl.fp8_w8a16_mm(x, it["qw"], it["sw"], y=y, stable_weights=True,
                                packed=self.packed)
            elif fl.quant_scaled_mm_preferred(it["M"], it["N"], it["K"], dynamic):
                fl.fp8_quant_scaled_mm(x, it["qw"], it["sw"], a_scale=it["sa"], dynamic=dynamic,
                                       out_scale=it.get("os"), y=y, ws=ws, stable_weights=True)
            else:
                fl.fp8_quant_per_tensor(x, q=it["qa"], scale=it["sa"], dynamic=dynamic, ws=ws)
                fl.fp8_scaled_mm(it["qa"], it["qw"], it["sa"], it["sw"], out_dtype=y.dtype,
                                 out_scale=it.get("os"), y=y, ws=ws, stable_weights=True)

        def serial():
            x_dev.copy_(x_host, non_blocking=True)
            for it, x, y in zip(items, xs, ys):
                product(it, x, y)
            y_host.copy_(y_dev, non_blocking=True)

        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in items]
        ev_done = [torch.cuda.Event() for _ in items]
        order = johnson_order([t.numel() for t in xd], [t.numel() for t in yd])

        def pipelined():
            comp = torch.cuda.current_stream(dev)
            s_in.wait_stream(comp)
            s_out.wait_stream(comp)
            with torch.cuda.stream(s_in):
                for i in order:
                    xd[i].copy_(xh[i], non_blocking=True)
                    ev_in[i].record(s_in)
            for i in order:
                it = items[i]
                comp.wait_event(ev_in[i])
                product(it, xs[i], ys[i])
                ev_done[i].record(comp)
                s_out.wait_event(ev_done[i])
                with torch.cuda.stream(s_out):
                    yh[i].copy_(yd[i], non_blocking=True)
            comp.wait_stream(s_in)
            comp.wait_stream(s_out)

        stream = torch.cuda.Stream(dev)

        def eager_time(body, n):
            with torch.cuda.stream(stream):
                t0 = time.perf_counter()
                for _ in range(n):
                    body()
                    stream.synchronize()
                return (time.perf_counter() - t0) / n

        def capture(body):
            with torch.cuda.stream(stream):
                for _ in range(3):
                    body()
                    stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                body()
            return g

        def graph_time(g, n):
            with torch.cuda.stream(stream):
                t0 = time.perf_counter()
                for _ in range(n):
                    g.replay()
                    stream.synchronize()
                return (time.perf_counter() - t0) / n

        g_pipe, g_serial = capture(pipelined), capture(serial)
        for g in (g_pipe, g_serial):
            graph_time(g, 3)
        # three interleaved rounds, the median of each form: the host link
        # and host memory are shared with the machine's other work
        n = max(3, steps // 3)
        rounds = [(graph_time(g_pipe, n), graph_time(g_serial, n), eager_time(pipelined, n))
                  for _ in range(3)]
        graph, graph_serial, eager = (sorted(r[i] for r in rounds)[1] for i in range(3))
        return graph, graph_serial, eager, h2d, d2h

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
            for i, (M, N, K) in self.shapes():
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
        for i, (M, N, K) in self.shapes():
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


SUSTAINED_AFTER_MS = 1000.0  # timed regions at least this long use the sustained tensor peak


def roofline(per_kind, peaks, ms_per_step, sustained=False):
    """Roofline of the dominant kernel: its algorithmic units per step over
    its time per step (the timed step time times its measured share).  A
    tensor-bound kernel timed inside a long run of steps (sustained=True,
    the timed region lasting SUSTAINED_AFTER_MS or more) is compared with the
    measured sustained bf16 rate x 2, one timed alone or briefly with the
    burst rate x 2; the fraction of the burst peak is reported in both
    cases."""
    if not per_kind:
        return None, None
    total = sum(v["ms"] for v in per_kind.values())
    kind, v = max(per_kind.items(), key=lambda kv: kv[1]["ms"])
    share = v["ms"] / total if total > 0 else 1.0
    secs = ms_per_step * share / 1e3
    ups = v["units_per_step"]
    if v["unit"] == "flops":
        achieved = ups / secs / 1e12
        burst = peaks["bf16_tflops"] * FP8_OVER_BF16
        which = "sustained" if sustained else "burst"
        base = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        peak = base * FP8_OVER_BF16
        rf = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
              "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
              "frac_of_burst": round(achieved / burst, 4)}
        rf["peak_source"] = (f"{peaks['source']} bf16 {which} {base} TFLOP/s x "
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
                  "scaled_mm_swapped": "gemm_swapab.cu", "scaled_mm_fused_quant": "gemm_swapab.cu",
                  "scaled_mm_fused_stream": "skinny_quant.cu",
                  "scaled_mm_tcgen05": "gemm_tcgen05.cu", "quant_dynamic": "quant.cu",
                  "quant_static": "quant.cu"}


def kernel_source_hash(src):
    """sha256 prefix of a kernel's translation unit followed by the library
    headers it includes, directly or through another one (a change to any of
    them invalidates a capture)."""
    csrc = os.path.join(ROOT, "fp8_quantized_linear_gb300", "csrc")
    order, todo = [], [src]
    while todo:
        name = todo.pop(0)
        if name in order or not os.path.exists(os.path.join(csrc, name)):
            continue
        order.append(name)
        with open(os.path.join(csrc, name)) as f:
            todo += re.findall(r'^#include "([^"]+)"', f.read(), flags=re.M)
    h = hashlib.sha256()
    for name in order:
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
    Workload.single_sm = args.single_sm_tiles
    work = Workload(args.workload, dev, packed_w8a16=args.w8a16_layout == "packed",
                    only_shape=args.only_shape)
    work.build()
    sampler = ClockSampler(dev)
    sampler.start()
    res = measure(work, args.steps, args.warmup, world)
    sampler.stop()
    clocks = sampler.summary(res["window"][1], res["window"][2])
    b, f = work.step_units()
    unit = work.headline_unit()
    value = aggregate(b if unit == "GB/s" else f, res["ms_per_step"], world, unit)
    rf, kinds = roofline(res["per_kind"], peaks, res["ms_per_step"],
                         sustained=res["ms_total"] >= SUSTAINED_AFTER_MS)
    # end to end through the public API with host buffers
    e2e_steps = max(9, min(args.steps, 60))
    dt_e2e, dt_serial, dt_eager, h2d, d2h = work.e2e(e2e_steps)

    def per_step(dt):
        return ((b / dt / 1e9) if unit == "GB/s" else (f / dt / 1e12)) * world
    e2e_val, e2e_serial, e2e_eager = per_step(dt_e2e), per_step(dt_serial), per_step(dt_eager)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(res["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 x e4m3 (fp32 accumulate)" if work.wl.kind == "w8a16"
                 else "e4m3 x e4m3 (fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": work.name, "description": work.wl.description,
                   "shapes": [list(s) for _, s in work.shapes()],
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
                "api": "per product: a pinned host->device copy of its activations on a copy "
                       "stream, its fp8_quantized_linear_gb300 call(s) on the compute stream once "
                       "that copy is done, a device->pinned host copy of its output on a second "
                       "copy stream once they are done; products in Johnson's-rule order on their "
                       "input and output copy bytes; captured in one CUDA graph, replayed and "
                       "synchronized once per step",
                "serial_value": round(e2e_serial, 3),
                "serial_api": "one copy of all activations, all calls, one copy of all outputs, "
                              "in one stream, one CUDA graph, synchronized per step",
                "eager_value": round(e2e_eager, 3),
                "eager_api": "the pipelined calls and copies issued eagerly, synchronized per step",
                "timing": f"host wall clock; each form in three interleaved rounds of "
                          f"{max(3, e2e_steps // 3)} steps, the median round"},
        "gpu_launches": res["gpu_launches"], "clocks": clocks,
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "source")},
    }
    if rank == 0:
        line["per_shape"] = per_shape(work, peaks, args.extra_steps)
        line["per_shape_timing"] = ("each product alone: a CUDA graph of the call on R rotating "
                                    "operand copies (together > 3x L2), replayed back to back "
                                    "between CUDA events; frac = achieved / min(tensor peak, "
                                    "HBM x AI)")
        jobs, units, desc = work.prepare_cpu_sample(1.0)
        secs = Workload.run_cpu_sample(jobs)
        cpu_val = (units / secs / 1e9) if unit == "GB/s" else (units / secs / 1e12)
        line["cpu_baseline"] = {"value": round(cpu_val, 6), "unit": unit, "cores": 1,
                                "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
        shapes = [(work.name, line["per_shape"])]
        entries = set(args.entries.split(",")) if args.entries else set()
        if not args.headline_only and work.name == HEADLINE:
            if "workloads" in entries:
                line["workloads"] = other_workloads(args, dev, peaks)
                shapes += [(e["workload"], e["per_shape"]) for e in line["workloads"]]
            if "norm_fusion" in entries:
                line["norm_fusion"] = norm_fusion_entry(dev, peaks, args.extra_steps)
            if "decode_block" in entries:
                line["decode_block"] = decode_block_entry(dev, peaks, args.extra_steps)
        line["small_m"] = small_m_summary(shapes)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def other_workloads(args, dev, peaks):
    """Short measurements of the other workloads (entries of the line)."""
    out = []
    for name in ENTRY_WORKLOADS:
        work = Workload(name, dev, packed_w8a16=args.w8a16_layout == "packed")
        work.build()
        res = measure(work, args.extra_steps, max(3, args.warmup // 2), 1)
        b, f = work.step_units()
        unit = work.headline_unit()
        sec = res["ms_per_step"] / 1e3
        rf, kinds = roofline(res["per_kind"], peaks, res["ms_per_step"])
        value = b / sec / 1e9 if unit == "GB/s" else f / sec / 1e12
        entry = {"workload": name, "value": round(value, 2), "unit": unit,
                 "ms_per_step": round(res["ms_per_step"], 4), "steps": args.extra_steps,
                 "roofline": rf, "kernels": kinds,
                 "per_shape": per_shape(work, peaks, args.extra_steps)}
        out.append(entry)
        del work
        torch.cuda.empty_cache()
    return out


def graph_time(fns, stream, reps):
    """Seconds per replay of a CUDA graph of the calls `fns`, replayed `reps`
    times back to back between two CUDA events on `stream`."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for fn in fns:
            fn()
    with torch.cuda.stream(stream):
        for _ in range(2):
            g.replay()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        b.synchronize()
    return a.elapsed_time(b) / 1e3 / reps


def norm_fusion_entry(dev, peaks, steps, eps=1e-5):
    """The prefill layer with its RMSNorm: per shape of the prefill workload
    (M = 1024, K = 4096, 1% outlier channels), RMSNorm with the dynamic
    per-tensor quantization fused into it (fp8_rmsnorm_quant) followed by the
    product, against the unfused layer: RMSNorm writing bf16
    (FP8L_NQ_NORM_ONLY), then the separate quantizer, then the product.
    Inputs rotate over copies larger than 3x L2."""
    import fp8_quantized_linear_gb300 as fl
    wl = synthetic.WORKLOADS["prefill_w8a8_outliers"]
    ws = fl.workspace(dev)
    stream = torch.cuda.Stream(dev)
    per_copy = sum(2 * M * K + M * K + N * K + 2 * M * N for (M, N, K) in wl.shapes)
    n_rot = max(1, min(16, math.ceil(3 * L2_BYTES / per_copy)))
    copies = []
    for r in range(n_rot):
        items = []
        for i, (M, N, K) in enumerate(wl.shapes):
            seed = wl.seed(i)
            x = synthetic.activation(M, K, wl.x_dtype, seed=seed, outlier_frac=wl.outlier_frac)
            w = synthetic.weight(N, K, torch.bfloat16, seed=seed).to(dev)
            qw, sw = fl.fp8_quant_per_tensor(w)
            items.append({"x": x.to(dev), "gamma": synthetic.norm_weight(K, wl.x_dtype, seed).to(dev),
                          "qw": qw, "sw": sw, "h": torch.empty((M, K), dtype=wl.x_dtype, device=dev),
                          "q": torch.empty((M, K), dtype=torch.uint8, device=dev),
                          "s": torch.empty(1, dtype=torch.float32, device=dev),
                          "y": torch.empty((M, N), dtype=torch.bfloat16, device=dev)})
            del w
        copies.append(items)

    def fused():
        return [lambda it=it: (fl.fp8_rmsnorm_quant(it["x"], it["gamma"], eps, q=it["q"],
                                                    scale=it["s"], ws=ws),
                               fl.fp8_scaled_mm(it["q"], it["qw"], it["s"], it["sw"], y=it["y"],
                                                ws=ws, stable_weights=True))
                for items in copies for it in items]

    def unfused():
        return [lambda it=it: (fl.fp8_rmsnorm_quant(it["x"], it["gamma"], eps, mode="norm_only",
                                                    h=it["h"]),
                               fl.fp8_quant_per_tensor(it["h"], q=it["q"], scale=it["s"], ws=ws),
                               fl.fp8_scaled_mm(it["q"], it["qw"], it["s"], it["sw"], y=it["y"],
                                                ws=ws, stable_weights=True))
                for items in copies for it in items]

    def norm_quant_only(fused_path):
        if fused_path:
            return [lambda it=it: fl.fp8_rmsnorm_quant(it["x"], it["gamma"], eps, q=it["q"],
                                                       scale=it["s"], ws=ws)
                    for items in copies for it in items]
        return [lambda it=it: (fl.fp8_rmsnorm_quant(it["x"], it["gamma"], eps, mode="norm_only",
                                                    h=it["h"]),
                               fl.fp8_quant_per_tensor(it["h"], q=it["q"], scale=it["s"], ws=ws))
                for items in copies for it in items]

    with torch.cuda.stream(stream):
        for fn in unfused() + fused():
            fn()
    stream.synchronize()
    reps = max(3, min(50, steps))
    t_f = graph_time(fused(), stream, reps) / n_rot
    t_u = graph_time(unfused(), stream, reps) / n_rot
    t_fq = graph_time(norm_quant_only(True), stream, reps) / n_rot
    t_uq = graph_time(norm_quant_only(False), stream, reps) / n_rot
    flops = sum(2 * M * N * K for (M, N, K) in wl.shapes)
    nq_bytes = sum(3 * M * K + 2 * K + 4 for (M, N, K) in wl.shapes)  # x read, codes written
    del copies
    torch.cuda.empty_cache()
    return {"workload": "prefill_w8a8_outliers with RMSNorm (eps 1e-5)",
            "fused_step_us": round(t_f * 1e6, 2), "unfused_step_us": round(t_u * 1e6, 2),
            "fused_TFLOP/s": round(flops / t_f / 1e12, 2),
            "unfused_TFLOP/s": round(flops / t_u / 1e12, 2),
            "speedup": round(t_u / t_f, 4),
            "norm_quant_us": {"fused": round(t_fq * 1e6, 2), "unfused": round(t_uq * 1e6, 2)},
            "fused_norm_quant_hbm_frac": round(nq_bytes / t_fq / 1e9 / peaks["hbm_gbs"], 4),
            "timing": f"CUDA graph per variant over {n_rot} rotating copies, {reps} replays"}


def decode_block_entry(dev, peaks, steps):
    """The Llama-3-8B-shaped decode layer (fused q/k/v, o, fused gate/up,
    down, each product reading the previous output) for M in {1, 16}: one
    CUDA graph per layer replayed back to back, against the same calls
    issued eagerly from Python.  Bytes per layer: the weights, scales and
    16-bit activations each product reads and writes (the W8A8 layer adds
    the quantizers' reads and writes)."""
    from fp8_quantized_linear_gb300.block import ORDER, SHAPES, DecodeBlock
    weights = {name: synthetic.weight(N, K, torch.bfloat16, seed=300 + i).to(dev)
               for i, (name, (N, K)) in enumerate(SHAPES.items())}
    stream = torch.cuda.Stream(dev)
    reps = max(10, min(200, steps * 10))
    out = []
    for kind in ("w8a16", "w8a8"):
        for M in (1, 16):
            blk = DecodeBlock(M, weights, kind=kind)
            blk.x.copy_(synthetic.activation(M, 4096, blk.act_dtype, seed=M).to(dev))
            g = blk.capture(stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(reps):
                    g.replay()
                e.record(stream)
                e.synchronize()
                t_graph = a.elapsed_time(e) / 1e3 / reps
                for _ in range(3):
                    blk.forward()
                stream.synchronize()
                t0 = time.perf_counter()
                a.record(stream)
                for _ in range(reps):
                    blk.forward()
                e.record(stream)
                e.synchronize()
                t_eager = (time.perf_counter() - t0) / reps
            nbytes = 0
            for name in ORDER:
                N, K = SHAPES[name]
                if kind == "w8a16":
                    nbytes += w8a16_bytes(M, N, K)
                else:
                    nbytes += w8a8_bytes(M, N, K, 2, True) + 3 * M * K
            out.append({"kind": kind, "M": M, "graph_us": round(t_graph * 1e6, 2),
                        "eager_us": round(t_eager * 1e6, 2),
                        "graph_speedup": round(t_eager / t_graph, 3),
                        "graph_GB/s": round(nbytes / t_graph / 1e9, 1),
                        "graph_hbm_frac": round(nbytes / t_graph / 1e9 / peaks["hbm_gbs"], 4),
                        "launches": blk.launches()})
            del blk
    del weights
    torch.cuda.empty_cache()
    return {"layer": "Llama-3-8B decode layer: qkv (6144,4096), o (4096,4096), gate_up "
                     "(28672,4096), down (4096,14336), chained",
            "timing": f"graph: {reps} replays between CUDA events; eager: the same calls from "
                      "Python, wall time per layer",
            "rows": out}


def shape_roofline(flops, nbytes, seconds, peak_tflops, hbm_gbs):
    """Figures of one product timed alone: achieved TFLOP/s and GB/s of
    algorithmic units, the roofline min(tensor peak, HBM x arithmetic
    intensity) with the bound that sets it, and the fractions of it and of
    HBM bandwidth."""
    tflops = flops / seconds / 1e12
    gbs = nbytes / seconds / 1e9
    mem_roof = hbm_gbs * (flops / nbytes) / 1e3  # TFLOP/s the bytes allow
    roof = min(peak_tflops, mem_roof)
    return {"TFLOP/s": round(tflops, 2), "GB/s": round(gbs, 1),
            "bound": "hbm" if mem_roof < peak_tflops else "tensor",
            "roof_TFLOP/s": round(roof, 1), "frac": round(tflops / roof, 4),
            "hbm_frac": round(gbs / hbm_gbs, 4)}


def per_shape(work, peaks, steps):
    """Every shape's product timed alone.  For each shape, a CUDA graph holds
    the one call on each of R copies of its operands (R such that the copies
    exceed three L2 sizes, so each call reads from HBM), and is replayed back
    to back between two CUDA events: no host dispatch or tensor-map encoding
    falls inside the timed window.  W8A8 shapes also time their activation
    quantization the same way, and the fused quantization + product where the
    step uses it (fused_us).  The roofline of each product is
    min(peak, HBM x AI): the FP8 tensor peak for W8A8, the 16-bit one for
    W8A16."""
    fl, wl, dev = work.fl, work.wl, work.device
    ws = fl.workspace(dev)
    stream = torch.cuda.Stream(dev)
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    reps = max(3, min(20, steps))
    rows = []

    def timed(fns):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for fn in fns:
                fn()
        with torch.cuda.stream(stream):
            g.replay()
            stream.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            b.synchronize()
        return a.elapsed_time(b) / 1e3 / (reps * len(fns))

    for base in work.copies[0]:
        M, N, K = base["M"], base["N"], base["K"]
        if wl.kind == "w8a16":
            nbytes, peak = w8a16_bytes(M, N, K), peaks["bf16_tflops"]
            kind = "w8a16_skinny"
        else:
            nbytes = w8a8_bytes(M, N, K, base["y"].element_size(), wl.w_scale == "channel")
            peak, kind = fp8_peak, W8A8_KINDS[fl.scaled_mm_kernel(M, N, K)]
        n_rot = max(1, min(64, math.ceil(3 * L2_BYTES / nbytes)))
        copies = [base] + [{k: (v.clone() if isinstance(v, torch.Tensor) else v)
                            for k, v in base.items()} for _ in range(n_rot - 1)]
        if wl.kind == "w8a16":
            prods = [lambda c=c: fl.fp8_w8a16_mm(c["x"], c["qw"], c["sw"], y=c["y"],
                                                 stable_weights=True, packed=work.packed)
                     for c in copies]
            quants, fuseds = [], []
        else:
            dyn = wl.act_scale == "dynamic"
            quants = [lambda c=c: fl.fp8_quant_per_tensor(c["x"], q=c["qa"], scale=c["sa"],
                                                          dynamic=dyn, ws=ws) for c in copies]
            prods = [lambda c=c: fl.fp8_scaled_mm(c["qa"], c["qw"], c["sa"], c["sw"],
                                                  out_dtype=c["y"].dtype, out_scale=c.get("os"),
                                                  y=c["y"], ws=ws, stable_weights=True,
                                                  single_sm=Workload.single_sm)
                     for c in copies]
            fuseds = ([lambda c=c: fl.fp8_quant_scaled_mm(c["x"], c["qw"], c["sw"], a_scale=c["sa"],
                                                          dynamic=dyn, out_scale=c.get("os"),
                                                          y=c["y"], ws=ws, stable_weights=True)
                       for c in copies] if fl.quant_scaled_mm_preferred(M, N, K, dyn) else [])
        with torch.cuda.stream(stream):  # eager pass: quantized activations, library set-up
            for fn in fuseds + quants + prods:
                fn()
        stream.synchronize()
        sec = timed(prods)
        row = {"M": M, "N": N, "K": K, "kernel": kind, "us": round(sec * 1e6, 2),
               **shape_roofline(2 * M * N * K, nbytes, sec, peak, peaks["hbm_gbs"]),
               "copies": n_rot}
        if quants:
            qsec = timed(quants)
            row["quant_us"] = round(qsec * 1e6, 2)
            row["quant_hbm_frac"] = round(3 * M * K / qsec / 1e9 / peaks["hbm_gbs"], 4)
        if fuseds:  # the call the step makes: quantization inside the product
            fsec = timed(fuseds)
            fb = fused_bytes(M, N, K, base["y"].element_size(), wl.w_scale == "channel")
            row["fused_us"] = round(fsec * 1e6, 2)
            row["fused_hbm_frac"] = round(fb / fsec / 1e9 / peaks["hbm_gbs"], 4)
        rows.append(row)
        del copies, prods, quants, fuseds
    torch.cuda.synchronize(dev)
    return rows


def small_m_summary(lines):
    """Which M <= 16 products reach HBM_TARGET of HBM bandwidth, timed alone."""
    hit, miss = [], []
    for wl_name, rows in lines:
        for r in rows:
            if r["M"] <= 16:
                (hit if r["hbm_frac"] >= HBM_TARGET else miss).append(
                    f"{wl_name} M={r['M']} N={r['N']} K={r['K']}: {r['hbm_frac']}")
    return {"target_hbm_frac": HBM_TARGET, "at_or_above": hit, "below": miss}


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
    work.shape_ids = (list(range(len(wl.shapes))) if args.only_shape is None
                      else [args.only_shape])
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
