"""GPU parity of the RMS normalization with the activation quantization
fused into it (fp8_rmsnorm_quant; "Condition to achieve linear speedup?":
the quantization fused into an element-wise kernel such as RMSNorm) against
the CPU oracle.

The normalized activations h are computed in float32 and rounded to the
16-bit format; they must equal the oracle's float64 RMSNorm rounded to that
format, except within a relative 2^-16 of a rounding midpoint, where either
neighbour is accepted (oracle.rounded_close).  Given h, the quantization is
the quantizer's: codes and scales must equal the oracle's quantization of
the kernel's own h bit for bit, and the codes must not depend on whether h
is written."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import DEV, assert_gemm_close, assert_status_ok, dev, host, sample_rows, scalar

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _inputs(M, K, dtype, seed, outliers=0.01):
    x = synthetic.activation(M, K, dtype, seed=seed, outlier_frac=outliers)
    gamma = synthetic.norm_weight(K, dtype, seed=seed)
    return x, gamma


def _check_h(h, x, gamma, dtype):
    res = oracle.rounded_close(host(h).astype(np.float64), oracle.rmsnorm_ref(x, gamma, EPS), dtype)
    assert res["ok"], res
    return res


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,K", [(1, 16), (3, 80), (7, 4096), (160, 4096), (300, 8192),
                                 (64, 14336), (16, 32768)])
@pytest.mark.parametrize("mode", ["dynamic", "static", "per_token", "norm_only"])
def test_modes_against_oracle(mode, M, K, dtype):
    x, gamma = _inputs(M, K, dtype, seed=M * 31 + K)
    xd, gd = dev(x), dev(gamma)
    s_static = scalar(0.0123) if mode == "static" else None
    q, s, h = fl.fp8_rmsnorm_quant(xd, gd, EPS, mode=mode, scale=s_static, want_h=True)
    _check_h(h, x, gamma, dtype)
    if mode == "norm_only":
        assert q is None
        return
    hh = host(h).astype(np.float32)
    if mode == "per_token":
        q_o, s_o = oracle.quant_per_row(hh)
    elif mode == "static":
        q_o, s_o = oracle.quant_per_tensor(hh, scale=np.float32(0.0123))
    else:
        q_o, s_o = oracle.quant_per_tensor(hh)
    assert np.array_equal(host(q), q_o)
    assert np.array_equal(host(s).reshape(-1).view(np.uint32),
                          np.asarray(s_o, np.float32).reshape(-1).view(np.uint32))
    # the same codes (and scales) when h is not written
    s2 = scalar(0.0123) if mode == "static" else None
    q2, s2, h2 = fl.fp8_rmsnorm_quant(xd, gd, EPS, mode=mode, scale=s2)
    assert h2 is None
    torch.cuda.synchronize()
    assert torch.equal(q2, q) and torch.equal(s2, s)


@pytest.mark.parametrize("M,K", [(1024, 4096), (8192, 4096), (4096, 8192)])
def test_dynamic_many_rows_per_block(M, K):
    # more rows per block than shared-memory stages: pass 2 re-reads rows
    x, gamma = _inputs(M, K, torch.bfloat16, seed=M + K)
    q, s, h = fl.fp8_rmsnorm_quant(dev(x), dev(gamma), EPS, mode="dynamic", want_h=True)
    _check_h(h, x, gamma, torch.bfloat16)
    q_o, s_o = oracle.quant_per_tensor(host(h).astype(np.float32))
    assert np.float32(host(s)[0]) == s_o
    assert np.array_equal(host(q), q_o)
    assert_status_ok()


def test_repeated_dynamic_calls_reuse_the_workspace():
    small, big = _inputs(5, 256, torch.bfloat16, 1), _inputs(2048, 4096, torch.bfloat16, 2)
    outs = []
    for x, gamma in (big, small, big, small, small):
        q, s, _ = fl.fp8_rmsnorm_quant(dev(x), dev(gamma), EPS)
        outs.append((host(q), host(s)[0]))
    assert np.array_equal(outs[0][0], outs[2][0]) and outs[0][1] == outs[2][1]
    assert np.array_equal(outs[1][0], outs[3][0]) and outs[1][1] == outs[4][1]
    # and the quantizer, which shares the barrier words, still agrees
    x, _ = small
    q, s = fl.fp8_quant_per_tensor(dev(x))
    q_o, s_o = oracle.quant_per_tensor(x)
    assert np.array_equal(host(q), q_o) and np.float32(host(s)[0]) == s_o
    assert_status_ok()


def test_empty_tensor_dynamic_scale_is_one():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    q, s, _ = fl.fp8_rmsnorm_quant(x, dev(torch.ones(64, dtype=torch.bfloat16)), EPS)
    assert host(s)[0] == 1.0


def test_norm_quant_then_product():
    # the prefill layer: fused norm + quantization, then the W8A8 product
    M, N, K = 1024, 4096, 4096
    x, gamma = _inputs(M, K, torch.bfloat16, seed=3)
    w = synthetic.weight(N, K, torch.bfloat16, seed=3)
    qw, sw = fl.fp8_quant_per_tensor(dev(w))
    q, s, h = fl.fp8_rmsnorm_quant(dev(x), dev(gamma), EPS, want_h=True)
    y = fl.fp8_scaled_mm(q, qw, s, sw, out_dtype=torch.bfloat16)
    rows = sample_rows(M, 64, seed=3)
    y_ref = oracle.scaled_mm_ref(host(q)[rows], host(qw), host(s)[0], host(sw))
    assert_gemm_close(host(y)[rows], y_ref)
    # unfused: norm-only, then the separate quantizer: the same codes
    _, _, h2 = fl.fp8_rmsnorm_quant(dev(x), dev(gamma), EPS, mode="norm_only")
    q2, s2 = fl.fp8_quant_per_tensor(h2)
    torch.cuda.synchronize()
    assert torch.equal(h2, h) and torch.equal(q2, q) and torch.equal(s2, s)
