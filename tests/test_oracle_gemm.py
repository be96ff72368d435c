"""Pins of the oracle's W8A8 scaled product and W8A16 weight-only product
("[Kernel][FP8] Initial support with dynamic per-tensor scaling", torch._scaled_mm;
"Marlin fp8", per-output-channel weight scale of shape [1, N])."""
import numpy as np
import pytest
import torch

import oracle
import pins
import synthetic


@pytest.fixture(scope="module")
def table():
    return oracle.decode_table()


def test_bruteforce_scaled_mm_pins(table):
    pins.check_scaled_mm(oracle.scaled_mm_bruteforce, table)


def test_matmul_scaled_mm_pins(table):
    pins.check_scaled_mm(oracle.scaled_mm_ref, table)


def test_bruteforce_scaled_mm_per_token_pins(table):
    pins.check_scaled_mm_per_token(oracle.scaled_mm_bruteforce, table)


def test_matmul_scaled_mm_per_token_pins(table):
    pins.check_scaled_mm_per_token(oracle.scaled_mm_ref, table)


@pytest.mark.parametrize("M,N,K", [(5, 48, 96), (17, 33, 80)])
def test_per_token_matmul_path_equals_loops(M, N, K):
    # per-token: one dynamic scale per activation row (the per-row quantizer)
    x = synthetic.activation(M, K, torch.bfloat16, seed=M * 11 + K, outlier_frac=0.01)
    qa, sa = oracle.quant_per_row(x)
    qw, sw = oracle.quant_per_row(synthetic.weight(N, K, torch.bfloat16, seed=N + 1))
    yb = oracle.scaled_mm_bruteforce(qa, qw, sa, sw)
    ym = oracle.scaled_mm_ref(qa, qw, sa, sw)
    assert np.allclose(ym, yb, rtol=1e-12, atol=1e-12 * np.abs(yb).max())


def test_per_token_scales_must_match_the_rows():
    qa = np.zeros((3, 16), np.uint8)
    qw = np.zeros((4, 16), np.uint8)
    with pytest.raises(ValueError):
        oracle.scaled_mm_ref(qa, qw, np.ones(2, np.float32), np.ones(4, np.float32))
    with pytest.raises(ValueError):
        oracle.scaled_mm_bruteforce(qa, qw, np.ones(4, np.float32), np.ones(4, np.float32))


def test_bruteforce_w8a16_pins(table):
    pins.check_w8a16(oracle.w8a16_bruteforce, table)


def test_matmul_w8a16_pins(table):
    pins.check_w8a16(oracle.w8a16_ref, table)


@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (5, 48, 96), (17, 33, 80), (16, 256, 512)])
@pytest.mark.parametrize("per_channel", [False, True])
def test_matmul_path_equals_loops(M, N, K, per_channel):
    # the float64 matrix product used for large shapes equals the triple loop
    x = synthetic.activation(M, K, torch.bfloat16, seed=M * 7 + K)
    w = synthetic.weight(N, K, torch.bfloat16, seed=N)
    qa, sa = oracle.quant_per_tensor(x)
    if per_channel:
        qw, sw = oracle.quant_per_row(w)
    else:
        qw, s = oracle.quant_per_tensor(w)
        sw = np.array([s], np.float32)
    yb = oracle.scaled_mm_bruteforce(qa, qw, sa, sw)
    ym = oracle.scaled_mm_ref(qa, qw, sa, sw)
    assert np.allclose(ym, yb, rtol=1e-12, atol=1e-12 * np.abs(yb).max())


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_w8a16_matmul_path_equals_loops(dtype):
    x = synthetic.activation(4, 160, dtype, seed=5)
    qw, sw = oracle.quant_per_row(synthetic.weight(40, 160, torch.bfloat16, seed=6))
    yb = oracle.w8a16_bruteforce(x, qw, sw)
    ym = oracle.w8a16_ref(x, qw, sw)
    assert np.allclose(ym, yb, rtol=1e-12, atol=1e-12 * np.abs(yb).max())


def test_quantized_product_tracks_unquantized(table):
    # sanity of the whole chain against the unquantized bf16 product: the
    # relative Frobenius error of an FP8 product of N(0,1)-like data is a few
    # percent (reported only; not a parity bound)
    x = synthetic.activation(16, 512, torch.bfloat16, seed=1000)
    w = synthetic.weight(256, 512, torch.bfloat16, seed=1000)
    qa, sa = oracle.quant_per_tensor(x)
    qw, s = oracle.quant_per_tensor(w)
    y = oracle.scaled_mm_ref(qa, qw, sa, np.array([s], np.float32))
    exact = x.double().numpy() @ w.double().numpy().T
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.1


def test_e4m3_output_ref():
    y = np.array([[448.0 * 0.5, -1.0, 0.0, 1e9]])
    codes = oracle.e4m3_output_ref(y, np.float32(0.5))
    assert list(codes[0]) == [0x7E, 0xC0, 0x00, 0x7E]
