"""Pins of the oracle's RMS normalization before the quantizer ("Condition
to achieve linear speedup?": the activation quantization fused into an
element-wise kernel such as RMSNorm; the plain Llama definition
h = x gamma / sqrt(mean x^2 + eps), stored in the activation's 16-bit
format, then quantized), of its rounding to the 16-bit formats, and of the
acceptance function for a 16-bit result computed in float32."""
import numpy as np
import pytest
import torch

import oracle
import pins


def test_rmsnorm_closed_forms():
    pins.check_rmsnorm(oracle.rmsnorm_ref)


def test_round_to_16bit_formats():
    pins.check_round_to(oracle.round_to)


def test_rounded_close():
    pins.check_rounded_close(oracle.rounded_close)


@pytest.mark.parametrize("mode", ["tensor", "row"])
def test_rmsnorm_quant_composition(mode):
    # the composition quantizes the rounded h exactly as the quantizer
    # quantizes any 16-bit tensor
    g = torch.Generator().manual_seed(9)
    x = torch.randn((6, 128), generator=g).to(torch.bfloat16)
    gamma = (torch.rand(128, generator=g) + 0.5).to(torch.bfloat16)
    q, s, h = oracle.rmsnorm_quant(x, gamma, 1e-5, mode=mode)
    assert np.array_equal(h, oracle.round_to(oracle.rmsnorm_ref(x, gamma, 1e-5), torch.bfloat16))
    hb = torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(hb.double(), torch.from_numpy(h))  # h holds bf16 values
    q2, s2 = (oracle.quant_per_row(hb) if mode == "row" else oracle.quant_per_tensor(hb))
    assert np.array_equal(q, q2) and np.array_equal(np.asarray(s), np.asarray(s2))


def test_constant_rows_quantize_to_the_largest_code():
    # h = +-1 everywhere (gamma = 1, eps = 0): scale 1/448, codes +-448
    x = torch.tensor([[2.0] * 32, [-0.5] * 32], dtype=torch.bfloat16)
    q, s, _ = oracle.rmsnorm_quant(x, torch.ones(32, dtype=torch.bfloat16), 0.0)
    assert np.float32(s) == np.float32(1.0) / np.float32(448.0)
    assert np.all(q[0] == 0x7E) and np.all(q[1] == 0xFE)
