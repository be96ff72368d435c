"""GPU parity of the per-token activation scales (FP8L_A_PER_TOKEN): one
activation scale per row of the E4M3 activations, in the epilogues of the
tcgen05 product (M > 16, persistent and cluster split-K) and of the
weight-streaming product (M <= 16), against the CPU oracle.  "RFC: FP8
Quantization Schema in vLLM", Scope, supports per-tensor scales and leaves
finer ones for later; this library reads the activation side of that as one
scale per token, as fp8_quant_per_row computes it."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import (DEV, assert_e4m3_close, assert_gemm_close, assert_status_ok, dev, host,
                      sample_rows, scalar)

pytestmark = pytest.mark.gpu

CODES = np.array([0x40, 0x38, 0x30, 0x00, 0xB0, 0xB8, 0xC0], np.uint8)  # -2 .. 2 as E4M3


@pytest.mark.parametrize("M", [1, 5, 16, 17, 64, 200, 300])
@pytest.mark.parametrize("per_channel", [False, True])
def test_exact_integer_distinct_row_scales(M, per_channel):
    # exact fp32 accumulation; distinct power-of-two row scales and column
    # scales with M != N: the output must be the rounded exact product bit
    # for bit, so a row scale taken from the wrong row or column shows
    rng = np.random.default_rng(M)
    N, K = 272, 1024
    qa = CODES[rng.integers(0, 7, (M, K))]
    qw = CODES[rng.integers(0, 7, (N, K))]
    sa = np.array([2.0 ** (m % 9 - 4) for m in range(M)], np.float32)
    sw = (np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32) if per_channel
          else np.array([0.375], np.float32))
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), dev(sa), dev(sw), out_dtype=torch.bfloat16,
                              per_token=True))
    exact = oracle.scaled_mm_bruteforce(qa, qw, sa, sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    bad = np.argwhere(y != want)
    assert bad.size == 0, (bad[:5], y[tuple(bad[0])], want[tuple(bad[0])])
    assert_status_ok()


@pytest.mark.parametrize("out", ["bf16", "fp16", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(3, 256, 512), (16, 4096, 4096), (64, 1024, 2048),
                                   (129, 272, 144), (1000, 2048, 1024)])
def test_full_path_per_token_quantization(M, N, K, out):
    # per-token quantization of the activations on the GPU (fp8_quant_per_row:
    # codes and scales bit-exact to the oracle), then the product
    x = synthetic.activation(M, K, torch.bfloat16, seed=M + N + K, outlier_frac=0.01)
    w = synthetic.weight(N, K, torch.bfloat16, seed=M + N + K)
    qa, sa = fl.fp8_quant_per_row(dev(x))
    qa_o, sa_o = oracle.quant_per_row(x)
    assert np.array_equal(host(qa), qa_o)
    assert np.array_equal(host(sa).view(np.uint32), sa_o.view(np.uint32))
    qw_o, sw_o = oracle.quant_per_row(w)
    rows = sample_rows(M, 64, seed=M)
    y_ref = oracle.scaled_mm_ref(qa_o[rows], qw_o, sa_o[rows], sw_o)
    if out == "e4m3":
        os_ = np.float32(np.abs(y_ref).max() / 448.0 * 0.8)
        y = fl.fp8_scaled_mm(qa, dev(qw_o), sa, dev(sw_o), out_dtype=torch.uint8,
                             out_scale=scalar(os_), per_token=True)
        assert_e4m3_close(host(y)[rows], y_ref, os_, (M, N, K))
    else:
        dt = torch.bfloat16 if out == "bf16" else torch.float16
        y = fl.fp8_scaled_mm(qa, dev(qw_o), sa, dev(sw_o), out_dtype=dt, per_token=True)
        assert_gemm_close(host(y)[rows], y_ref, (M, N, K, out))
    assert_status_ok()


def test_one_scale_for_every_row_equals_per_tensor():
    M, N, K = 300, 512, 768
    rng = np.random.default_rng(5)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(finite, size=(M, K)).astype(np.uint8)
    qw = rng.choice(finite, size=(N, K)).astype(np.uint8)
    sw = np.array([0.01], np.float32)
    y_pt = fl.fp8_scaled_mm(dev(qa), dev(qw), dev(np.full(M, 0.02, np.float32)), dev(sw),
                            out_dtype=torch.bfloat16, per_token=True)
    y_t = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.02), dev(sw), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(y_pt, y_t)
