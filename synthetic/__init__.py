"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws random numbers and lists workload shapes.  It holds none of
the layer's arithmetic (no scale, no cast, no product), so both the GPU path
and the CPU oracle can take their inputs from it without sharing method code.

Every tensor is drawn in float32 on the CPU with ``torch.Generator`` and then
rounded to its storage dtype, so the oracle and the GPU receive identical bytes.
Large matrices are drawn in blocks of rows with one seed per block, so that a
test can regenerate only the rows it samples.

Workloads are Llama-shaped linear layers (nn.Linear layout: W is [N, K], X is
[M, K]).  Activations are N(0, 1); weights are N(0, 0.02).  The prefill
workload has 1% of its K channels scaled by 50 (activation outlier channels).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

ROW_BLOCK = 1024


def _block_seed(seed: int, block: int) -> int:
    return (int(seed) * 1_000_003 + 7919 * int(block) + 12345) % (2 ** 63 - 1)


def normal_matrix(rows: int, cols: int, std: float, dtype: torch.dtype,
                  seed: int, row_subset=None) -> torch.Tensor:
    """[rows, cols] (or [len(row_subset), cols]) CPU tensor, N(0, std^2) drawn
    in float32 block by block, then rounded to ``dtype``."""
    if row_subset is None:
        out = torch.empty((rows, cols), dtype=dtype)
        for b0 in range(0, rows, ROW_BLOCK):
            nb = min(ROW_BLOCK, rows - b0)
            g = torch.Generator().manual_seed(_block_seed(seed, b0 // ROW_BLOCK))
            blk = torch.randn((nb, cols), generator=g, dtype=torch.float32)
            out[b0:b0 + nb] = (blk * std).to(dtype)
        return out
    idx = torch.as_tensor(row_subset, dtype=torch.int64)
    out = torch.empty((idx.numel(), cols), dtype=dtype)
    cache = {}
    for i, r in enumerate(idx.tolist()):
        if not 0 <= r < rows:
            raise IndexError(r)
        b = r // ROW_BLOCK
        if b not in cache:
            nb = min(ROW_BLOCK, rows - b * ROW_BLOCK)
            g = torch.Generator().manual_seed(_block_seed(seed, b))
            cache[b] = torch.randn((nb, cols), generator=g, dtype=torch.float32)
        out[i] = (cache[b][r - b * ROW_BLOCK] * std).to(dtype)
    return out


def outlier_channels(K: int, seed: int, frac: float = 0.01) -> torch.Tensor:
    """ceil(frac*K) distinct channel indices chosen by a seeded permutation."""
    g = torch.Generator().manual_seed(_block_seed(seed, 999_983))
    return torch.randperm(K, generator=g)[: int(math.ceil(frac * K))]


def activation(M: int, K: int, dtype: torch.dtype, seed: int,
               outlier_frac: float = 0.0, outlier_gain: float = 50.0,
               row_subset=None) -> torch.Tensor:
    """X ~ N(0,1) [M, K]; optionally a fraction of K channels scaled by
    ``outlier_gain`` before rounding to ``dtype``."""
    x = normal_matrix(M, K, 1.0, torch.float32, seed, row_subset=row_subset)
    if outlier_frac > 0:
        ch = outlier_channels(K, seed, outlier_frac)
        x[:, ch] *= outlier_gain
    return x.to(dtype)


def weight(N: int, K: int, dtype: torch.dtype, seed: int,
           row_subset=None) -> torch.Tensor:
    """W ~ N(0, 0.02^2) [N, K]."""
    return normal_matrix(N, K, 0.02, dtype, seed + 500_000, row_subset=row_subset)


def norm_weight(K: int, dtype: torch.dtype, seed: int) -> torch.Tensor:
    """RMSNorm gain gamma [K] ~ N(1, 0.1^2)."""
    g = torch.Generator().manual_seed(_block_seed(seed, 777_777))
    return (1.0 + 0.1 * torch.randn(K, generator=g, dtype=torch.float32)).to(dtype)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                     # 1-based position in the workload list
    description: str
    shapes: tuple                  # ((M, N, K), ...)
    x_dtype: torch.dtype
    act_scale: str                 # "dynamic" | "static" | "none" (W8A16)
    w_scale: str                   # "tensor" | "channel"
    out_dtype: str                 # "bf16" | "fp16" | "e4m3"
    outlier_frac: float = 0.0
    kind: str = "w8a8"             # "w8a8" | "w8a16"
    extra: dict = field(default_factory=dict)

    def seed(self, shape_idx: int) -> int:
        return 1000 * self.index + shape_idx


def _grid(nk, ms):
    return tuple((m, n, k) for (n, k) in nk for m in ms)


WORKLOADS = {
    w.name: w for w in [
        Workload(
            "tiny_w8a8", 1,
            "X bf16 [16,512] ~N(0,1), W bf16 [256,512] ~N(0,0.02); dynamic "
            "per-tensor activation scale, per-tensor weight scale, bf16 out",
            ((16, 256, 512),), torch.bfloat16, "dynamic", "tensor", "bf16"),
        Workload(
            "decode_w8a16", 2,
            "fp16 X [M in {1,4,16}, K] ~N(0,1) times FP8 W ~N(0,0.02) with a "
            "per-channel fp32 scale; (N,K) in {(12288,4096),(4096,4096),"
            "(22016,4096),(4096,11008)}",
            _grid(((12288, 4096), (4096, 4096), (22016, 4096), (4096, 11008)),
                  (1, 4, 16)),
            torch.float16, "none", "channel", "fp16", kind="w8a16"),
        Workload(
            "prefill_w8a8_outliers", 3,
            "M=1024, (N,K) in {(4096,4096),(11008,4096)}; X bf16 ~N(0,1) with "
            "1% of K channels x50; W ~N(0,0.02); dynamic per-tensor scales, "
            "bf16 out",
            _grid(((4096, 4096), (11008, 4096)), (1024,)),
            torch.bfloat16, "dynamic", "tensor", "bf16", outlier_frac=0.01),
        Workload(
            "llama3_8b_w8a8_sweep", 4,
            "(N,K) in {(6144,4096),(4096,4096),(28672,4096),(4096,14336)} x "
            "M in {1,16,128,1024,8192}; bf16 in/out; dynamic per-tensor scales",
            _grid(((6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336)),
                  (1, 16, 128, 1024, 8192)),
            torch.bfloat16, "dynamic", "tensor", "bf16"),
        Workload(
            "llama70b_static_fp8out", 5,
            "(N,K) in {(10240,8192),(8192,8192),(57344,8192),(8192,28672)} x "
            "M in {1,64,1024,4096}; static input scale, per-channel weight "
            "scale, E4M3 output through output_scale",
            _grid(((10240, 8192), (8192, 8192), (57344, 8192), (8192, 28672)),
                  (1, 64, 1024, 4096)),
            torch.bfloat16, "static", "channel", "e4m3"),
    ]
}


def calibration_seed(seed: int) -> int:
    """Seed of the independent calibration draw behind a static scale."""
    return seed + 500
