"""A Llama-3-8B-shaped decode layer of FP8 linear products, chained and
captured in one CUDA graph.

"Marlin fp8" measures decode latency at batch size 1: FP8 weights win only
once the step runs with CUDA graphs and a static cache (8.83 against 12.28
ms/token for fp16 on A100), while eagerly launched FP8 loses (33.87 against
32.11 ms).  This module chains the layer's four products at the model's
shapes, each consuming the previous one's output, so a whole layer's launches
can be replayed from one graph and timed against issuing them eagerly.

Shapes (nn.Linear [N, K], hidden 4096): fused q/k/v (6144, 4096), o
(4096, 4096), fused gate/up (28672, 4096), down (4096, 14336).  Attention and
the SiLU gate are not part of this path: the o product reads the first
M x 4096 values of the q/k/v output, and the down product the first
M x 14336 values of the gate/up output, as [M, K] tensors (stand-ins that keep
each product's input a function of the previous output).

  * "w8a16": fp16 activations times E4M3 weights with per-channel scales
    (fp8_w8a16_mm), the decode path; weights packed at set-up.
  * "w8a8": bf16 activations; RMSNorm fused with the dynamic per-tensor
    quantization before q/k/v (fp8_rmsnorm_quant) and the W8A8 product
    (fp8_scaled_mm) with per-channel weight scales, bf16 outputs; before o,
    gate/up and down the dynamic quantization runs inside the product
    (fp8_quant_scaled_mm) where quant_scaled_mm_preferred says that is the
    faster way (a few tokens), else as its own launch
    (fp8_quant_per_tensor).

Every call goes through the binding to the library's kernels; this module
only owns the buffers and the order of the calls.
"""
from __future__ import annotations

import torch

from . import _binding as b

HIDDEN = 4096
SHAPES = {"qkv": (6144, 4096), "o": (4096, 4096), "gate_up": (28672, 4096),
          "down": (4096, 14336)}
ORDER = ("qkv", "o", "gate_up", "down")


class DecodeBlock:
    """One decode layer for `M` tokens.  weights: {name: bf16 [N, K] tensor}
    on the device (quantized per channel at construction)."""

    def __init__(self, M: int, weights: dict, kind: str = "w8a16", eps: float = 1e-5,
                 gamma: torch.Tensor | None = None):
        if kind not in ("w8a16", "w8a8"):
            raise ValueError(kind)
        self.M, self.kind, self.eps = M, kind, eps
        dev = weights["qkv"].device
        self.device = dev
        self.act_dtype = torch.float16 if kind == "w8a16" else torch.bfloat16
        self.w, self.sw = {}, {}
        for name in ORDER:
            N, K = SHAPES[name]
            assert tuple(weights[name].shape) == (N, K)
            q, s = b.fp8_quant_per_row(weights[name])
            self.w[name] = b.fp8_pack_w8a16_weights(q) if kind == "w8a16" else q
            self.sw[name] = s
        self.x = torch.zeros((M, HIDDEN), dtype=self.act_dtype, device=dev)
        self.y = {name: torch.empty((M, SHAPES[name][0]), dtype=self.act_dtype, device=dev)
                  for name in ORDER}
        if kind == "w8a8":
            self.gamma = (gamma if gamma is not None
                          else torch.ones(HIDDEN, dtype=self.act_dtype, device=dev))
            self.qa = {name: torch.empty((M, SHAPES[name][1]), dtype=torch.uint8, device=dev)
                       for name in ORDER}
            self.sa = {name: torch.empty(1, dtype=torch.float32, device=dev) for name in ORDER}
            self.ws = b.workspace(dev)
        self.graph = None

    def input_of(self, name: str) -> torch.Tensor:
        """The [M, K] input of a product: x for q/k/v, else the leading
        M x K values of the previous product's output."""
        K = SHAPES[name][1]
        if name == "qkv":
            return self.x
        prev = ORDER[ORDER.index(name) - 1]
        return self.y[prev].view(-1)[: self.M * K].view(self.M, K)

    def forward(self) -> torch.Tensor:
        """Issues the layer's calls on the current stream; returns the down
        product's output buffer."""
        for name in ORDER:
            inp = self.input_of(name)
            if self.kind == "w8a16":
                b.fp8_w8a16_mm(inp, self.w[name], self.sw[name], y=self.y[name],
                               stable_weights=True, packed=True)
                continue
            if name == "qkv":
                b.fp8_rmsnorm_quant(inp, self.gamma, self.eps, q=self.qa[name],
                                    scale=self.sa[name], ws=self.ws)
            elif self.fused(name):
                b.fp8_quant_scaled_mm(inp, self.w[name], self.sw[name], a_scale=self.sa[name],
                                      dynamic=True, out_dtype=self.act_dtype, y=self.y[name],
                                      ws=self.ws, stable_weights=True)
                continue
            else:
                b.fp8_quant_per_tensor(inp, q=self.qa[name], scale=self.sa[name], ws=self.ws)
            b.fp8_scaled_mm(self.qa[name], self.w[name], self.sa[name], self.sw[name],
                            out_dtype=self.act_dtype, y=self.y[name], ws=self.ws,
                            stable_weights=True)
        return self.y["down"]

    def fused(self, name: str) -> bool:
        """Whether the product `name` runs with its quantization fused (W8A8,
        not q/k/v, where quant_scaled_mm_preferred says the fused call is the
        faster one)."""
        N, K = SHAPES[name]
        return (self.kind == "w8a8" and name != "qkv" and
                b.quant_scaled_mm_preferred(self.M, N, K, dynamic=True))

    def launches(self) -> int:
        """Kernel launches of one forward()."""
        if self.kind == "w8a16":
            return 4
        return sum(1 if self.fused(n) else 2 for n in ORDER)

    def capture(self, stream: torch.cuda.Stream | None = None) -> torch.cuda.CUDAGraph:
        """Runs forward() once eagerly (library set-up outside the capture),
        then captures it into a CUDA graph kept on the object."""
        stream = stream or torch.cuda.Stream(self.device)
        with torch.cuda.stream(stream):
            self.forward()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.forward()
        self.graph = g
        return g
