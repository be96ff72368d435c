"""GPU parity of the two tile shapes of the tcgen05 product: 256 x 256 tiles
spanning a pair of SMs (tcgen05.mma.cta_group::2, the default when the
product has enough tiles; the columns left after the last whole round of
tiles run as narrower tail tiles) and 128 x 256 tiles on one SM each
(FP8L_SINGLE_SM_TILES).  Both against the CPU oracle: exact-integer products
bit for bit, permutation weights exactly, and Gaussian operands within the
layer's tolerance, with ragged M and N tails of the 256-row pair tiles."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import (assert_e4m3_close, assert_gemm_close, assert_status_ok, dev, host,
                      sample_rows, scalar, scaled_mm_ref_rows)

pytestmark = pytest.mark.gpu

CODES = np.array([0x40, 0x38, 0x30, 0x00, 0xB0, 0xB8, 0xC0], np.uint8)  # -2 .. 2 as E4M3


@pytest.mark.parametrize("single_sm", [False, True])
@pytest.mark.parametrize("M,N,K", [(1280, 2048, 1024), (1000, 2320, 640), (2304, 4096, 2048),
                                   (4097, 1040, 384)])
def test_exact_integer(M, N, K, single_sm):
    rng = np.random.default_rng(M + N + K)
    qa = CODES[rng.integers(0, 7, (M, K))]
    qw = CODES[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16,
                              single_sm=single_sm))
    rows = sample_rows(M, 160, seed=M)
    exact = oracle.scaled_mm_ref(qa[rows], qw, np.float32(0.5), sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    bad = np.argwhere(y[rows] != want)
    assert bad.size == 0, (bad[:5],)
    assert_status_ok()


# the pair kernel's tile plans: 256 x 256 tiles in whole rounds, then the
# left-over columns as narrower tiles (widths 96, 128, 192 and 224 here,
# and 224 throughout when the tiles are fewer than the SM pairs), with
# ragged ends of N inside the last tail tile
@pytest.mark.parametrize("M,N,K", [(1024, 10240, 256), (1024, 8192, 384), (1024, 4096, 512),
                                   (4096, 10240, 128), (4096, 8192, 128), (1000, 11008, 256),
                                   (4097, 1040, 384)])
def test_tail_tiles_exact_integer(M, N, K):
    rng = np.random.default_rng(M * 3 + N + K)
    qa = CODES[rng.integers(0, 7, (M, K))]
    qw = CODES[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16))
    rows = sample_rows(M, 96, seed=N)
    exact = oracle.scaled_mm_ref(qa[rows], qw, np.float32(0.5), sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    bad = np.argwhere(y[rows] != want)
    assert bad.size == 0, (bad[:5],)
    assert_status_ok()


@pytest.mark.parametrize("single_sm", [False, True])
def test_permutation_weights(single_sm):
    K = N = 1024
    M = 3072  # 96 single-SM tiles: enough for the pair kernel (no split-K)
    pi = (np.arange(N) * 389 + 11) % K
    qw = np.zeros((N, K), np.uint8)
    qw[np.arange(N), pi] = 0x38
    rng = np.random.default_rng(6)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(finite, size=(M, K)).astype(np.uint8)
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16,
                              single_sm=single_sm))
    want = oracle.decode_table()[qa][:, pi] * 0.5 * sw[None, :]
    want = torch.from_numpy(want).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y, want)


@pytest.mark.parametrize("out", ["bf16", "fp16", "e4m3"])
@pytest.mark.parametrize("per_token", [False, True])
def test_gaussian_operands(out, per_token):
    M, N, K = 2000, 3072, 4096
    x = synthetic.activation(M, K, torch.bfloat16, seed=77, outlier_frac=0.01)
    w = synthetic.weight(N, K, torch.bfloat16, seed=77)
    qa, sa = (oracle.quant_per_row(x) if per_token else oracle.quant_per_tensor(x))
    qw, sw = oracle.quant_per_row(w)
    rows = sample_rows(M, 96, seed=3)
    y_ref = scaled_mm_ref_rows(qa[rows], qw, sa[rows] if per_token else sa, sw)
    sa_d = dev(np.atleast_1d(np.asarray(sa, np.float32)))
    if out == "e4m3":
        os_ = np.float32(np.abs(y_ref).max() / 448.0 * 0.8)
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), sa_d, dev(sw), out_dtype=torch.uint8,
                             out_scale=scalar(os_), per_token=per_token)
        assert_e4m3_close(host(y)[rows], y_ref, os_)
    else:
        dt = torch.bfloat16 if out == "bf16" else torch.float16
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), sa_d, dev(sw), out_dtype=dt, per_token=per_token)
        assert_gemm_close(host(y)[rows], y_ref)
    assert_status_ok()


def test_pair_and_single_tiles_agree():
    # the same product through both tile shapes; reported, and within the
    # tolerance of each other
    M, N, K = 3000, 5120, 2048
    rng = np.random.default_rng(12)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(finite, size=(M, K)).astype(np.uint8)
    qw = rng.choice(finite, size=(N, K)).astype(np.uint8)
    a, w, s1, s2 = dev(qa), dev(qw), scalar(1e-3), scalar(1e-3)
    y2 = fl.fp8_scaled_mm(a, w, s1, s2, out_dtype=torch.float16)
    y1 = fl.fp8_scaled_mm(a, w, s1, s2, out_dtype=torch.float16, single_sm=True)
    assert_gemm_close(host(y2), host(y1).astype(np.float64))
