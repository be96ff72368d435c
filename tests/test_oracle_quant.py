"""Pins of the oracle's per-tensor and per-row quantization ("[Kernel][FP8]
Initial support with dynamic per-tensor scaling", Algorithm; "RFC: FP8
Quantization Schema in vLLM", static input scale)."""
import numpy as np
import pytest
import torch

import oracle
import pins
import synthetic


@pytest.fixture(scope="module")
def table():
    return oracle.decode_table()


def test_worked_examples():
    pins.check_quant_worked(oracle.quant_per_tensor)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("outliers", [0.0, 0.01])
def test_invariants(table, dtype, outliers):
    x = synthetic.activation(64, 384, dtype, seed=17, outlier_frac=outliers)
    pins.check_quant_invariants(oracle.quant_per_tensor, table, x)


def test_invariants_tiny_values(table):
    # amax small enough that many codes are E4M3 subnormals
    g = torch.Generator().manual_seed(2)
    x = (torch.randn(4000, generator=g) * torch.exp2(torch.randint(-20, 0, (4000,), generator=g).float()))
    pins.check_quant_invariants(oracle.quant_per_tensor, table, x.to(torch.bfloat16))


def test_zero_tensor(table):
    pins.check_quant_invariants(oracle.quant_per_tensor, table, torch.zeros(37, dtype=torch.bfloat16))
    q, s = oracle.quant_per_tensor(torch.zeros(5, dtype=torch.float16))
    assert s == np.float32(1.0) and not q.any()


def test_negative_zero_codes():
    x = torch.tensor([-0.0, -1e-6, 100.0], dtype=torch.float32)
    q, _ = oracle.quant_per_tensor(x)
    assert list(q) == [0x80, 0x80, 0x7E]


def test_static_scale():
    pins.check_quant_static(oracle.quant_per_tensor, oracle.e4m3_encode)


def test_per_row(table):
    w = synthetic.weight(12, 64, torch.bfloat16, seed=3)
    w[5] = 0
    q, s = oracle.quant_per_row(w)
    assert q.shape == (12, 64) and s.shape == (12,)
    for r in range(12):
        pins.check_quant_invariants(oracle.quant_per_tensor, table, w[r])
        qr, sr = oracle.quant_per_tensor(w[r])
        assert np.array_equal(qr, q[r]) and sr == s[r]
    assert s[5] == 1.0 and not q[5].any()
