"""FP8 E4M3 quantized linear layer for NVIDIA GB300 (sm_103a).

A C-ABI library (``libfp8linear.so``, declared in ``include/fp8linear.h``)
with hand-written CUDA kernels, and a thin ctypes binding whose functions
carry the C entry points' names:

  fp8_quant_per_tensor  dynamic or static per-tensor quantization to E4M3
  fp8_quant_per_row     per-row quantization (weights at setup; per-token activations)
  fp8_rmsnorm_quant     RMSNorm with the activation quantization fused into it
  fp8_scaled_mm         W8A8 scaled product (tcgen05 products; few tokens and
                        small weights streamed on the CUDA cores)
  fp8_quant_scaled_mm   the same for up to 128 tokens of 16-bit x, its per-tensor
                        quantization (dynamic or static scale) fused into the product
  quant_scaled_mm_preferred  whether that fused call is the faster way for a shape
  scaled_mm_kernel      which of the three kernels fp8_scaled_mm runs for a shape
  w8a16_mm_kernel       which of the two kernels fp8_w8a16_mm runs
  fp8_grouped_mm        W8A8 products of mixture-of-experts layers (device offsets)
  fp8_w8a16_mm          weight-only fp16/bf16 x E4M3 product
  fp8_pack_w8a16_weights  weights permuted once into the order that product
                          reads them (fragment order, contiguous per CTA)

The library is loaded on first use; nothing here computes on the CPU.
"""
from ._binding import (  # noqa: F401
    BF16, E4M3, F16, F32, Fp8LinearError, LIB_PATH, fp8_grouped_mm, fp8_pack_w8a16_weights,
    fp8_packed_weight_bytes, fp8_quant_per_row, fp8_quant_per_tensor, fp8_quant_scaled_mm,
    fp8_scaled_mm, quant_scaled_mm_preferred,
    fp8_rmsnorm_quant, fp8_w8a16_mm, fp8l_debug_waits, fp8l_read_status, fp8l_workspace_bytes, load,
    scaled_mm_kernel, strerror, w8a16_mm_kernel, workspace)
