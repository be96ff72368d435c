"""GPU parity of the W8A16 tcgen05 product (fp8_w8a16_mm with
FP8L_KERNEL_SWAPPED, the automatic choice from 17 to 64 tokens): E4M3 weights
widened to the activations' 16-bit type in tensor memory, 128 weight rows by
the tokens per tile, clusters splitting K when the weight blocks are few.
Against the CPU oracle ("Marlin fp8": y = w_scale[n] sum_k x dec(w)):
exact-integer products bit for bit in both weight layouts and both 16-bit
types (ragged N and K tails, one partial k-block, every split the launcher
picks), every E4M3 code through the widening, the decode workload's shapes
within the layer's tolerance, agreement with the CUDA-core kernel, and a
graph-captured chain of programmatic dependents."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import DEV, assert_gemm_close, dev, host

pytestmark = pytest.mark.gpu

CODES = np.array([0x40, 0x38, 0x30, 0x00, 0xB0, 0xB8, 0xC0], np.uint8)  # -2 .. 2 as E4M3


def _status_ok():
    st = fl.fp8l_read_status(fl.workspace(DEV))
    assert st == 0, fl.strerror(st)


def _mm(x, qw, sw, packed, **kw):
    w = fl.fp8_pack_w8a16_weights(dev(qw)) if packed else dev(qw)
    return fl.fp8_w8a16_mm(dev(x), w, dev(sw), packed=packed, kernel="swapped", **kw)


# N = 16: one partial weight block (split up to 8); 2320: a ragged last
# block; 4096 and 12288: splits 8 and 3.  K = 16: one partial k-block; 80: a
# ragged second one; 4096: 32 k-blocks; 11008: 86, split in uneven shares.
@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("xdtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M", [1, 9, 16, 17, 64])
@pytest.mark.parametrize("N,K", [(16, 80), (2320, 640), (4096, 4096), (12288, 16), (4096, 11008)])
def test_exact_integer(M, N, K, xdtype, packed):
    rng = np.random.default_rng(M * 31 + N + K)
    qw = CODES[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    x = torch.from_numpy(rng.integers(-3, 4, (M, K)).astype(np.float32) / 2).to(xdtype)
    y = host(_mm(x, qw, sw, packed))
    exact = oracle.w8a16_ref(x, qw, sw)  # every partial sum is exact
    want = torch.from_numpy(exact).to(xdtype).float().numpy()
    bad = np.argwhere(y != want)
    assert bad.size == 0, (bad[:5], y[tuple(bad[0])], want[tuple(bad[0])])
    _status_ok()


@pytest.mark.parametrize("xdtype", [torch.float16, torch.bfloat16])
def test_every_code_widens_exactly(xdtype):
    # channel n holds code n at one k position and zeros elsewhere, x is all
    # ones: y[:, n] = sw[n] * dec(n) exactly, for every finite code (the
    # subnormals 0x01-0x07, both zeros, the largest 0x7E and 0xFE)
    N, K, M = 256, 128, 16
    codes = np.arange(256, dtype=np.uint8)
    codes[[0x7F, 0xFF]] = 0x00  # NaN codes are outside the contract
    qw = np.zeros((N, K), np.uint8)
    qw[np.arange(N), (np.arange(N) * 5) % K] = codes
    sw = np.array([2.0 ** (n % 3 - 1) for n in range(N)], np.float32)
    x = torch.ones((M, K), dtype=xdtype)
    for packed in (False, True):
        y = host(_mm(x, qw, sw, packed))
        want = oracle.decode_table()[codes] * sw.astype(np.float64)
        want = torch.from_numpy(np.broadcast_to(want, (M, N)).copy()).to(xdtype).float().numpy()
        assert np.array_equal(y, want), (packed, np.argwhere(y != want)[:5])


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("xdtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("nk", [(12288, 4096), (4096, 4096), (22016, 4096), (4096, 11008)])
def test_decode_shapes(nk, xdtype, packed):
    N, K = nk
    M = 16
    x = synthetic.activation(M, K, xdtype, seed=N + K)
    qw, sw = oracle.quant_per_row(synthetic.weight(N, K, torch.bfloat16, seed=N))
    y = host(_mm(x, qw, sw, packed, stable_weights=True))
    assert_gemm_close(y, oracle.w8a16_ref(x, qw, sw), (N, K, xdtype, packed))
    _status_ok()


@pytest.mark.parametrize("M", [9, 16, 40])
def test_agrees_with_cuda_core_kernel(M):
    # exact-integer operands: both kernels give the exact value rounded once
    N, K = 3072, 2048
    rng = np.random.default_rng(M)
    qw = CODES[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    x = torch.from_numpy(rng.integers(-4, 5, (M, K)).astype(np.float32)).to(torch.float16)
    xd, wd, sd = dev(x), dev(qw), dev(sw)
    y_tc = host(fl.fp8_w8a16_mm(xd, wd, sd, kernel="swapped"))
    y_cc = host(fl.fp8_w8a16_mm(xd, wd, sd, kernel="stream"))
    assert np.array_equal(y_tc, y_cc)


def test_graph_chain_with_stable_weights():
    # x -> y1 = x W1^T -> y2 = y1 W2^T in one CUDA graph, both products
    # programmatic dependents that load weights before their wait; outputs
    # zeroed before every replay
    M, K, N = 16, 4096, 4096
    x = synthetic.activation(M, K, torch.float16, seed=71)
    q1, s1 = oracle.quant_per_row(synthetic.weight(N, K, torch.bfloat16, seed=72))
    q2, s2 = oracle.quant_per_row(synthetic.weight(N, N, torch.bfloat16, seed=73))
    xd = dev(x)
    w1 = fl.fp8_pack_w8a16_weights(dev(q1))
    w2 = dev(q2)
    s1d, s2d = dev(s1), dev(s2)
    y1 = torch.empty((M, N), dtype=torch.float16, device=DEV)
    y2 = torch.empty((M, N), dtype=torch.float16, device=DEV)

    def step():
        fl.fp8_w8a16_mm(xd, w1, s1d, y=y1, packed=True, stable_weights=True, kernel="swapped")
        fl.fp8_w8a16_mm(y1, w2, s2d, y=y2, stable_weights=True, kernel="swapped")

    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(3):
        y1.zero_()
        y2.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert_gemm_close(host(y1), oracle.w8a16_ref(x, q1, s1))
    y1h = torch.from_numpy(host(y1)).to(torch.float16)
    assert_gemm_close(host(y2), oracle.w8a16_ref(y1h, q2, s2))
    _status_ok()


def test_bounds():
    x = torch.zeros((65, 64), dtype=torch.float16, device=DEV)
    w = torch.zeros((64, 64), dtype=torch.uint8, device=DEV)
    s = torch.ones(64, dtype=torch.float32, device=DEV)
    with pytest.raises(RuntimeError):
        fl.fp8_w8a16_mm(x, w, s, kernel="swapped")
    y = fl.fp8_w8a16_mm(x[:0], w, s, kernel="swapped")
    assert y.shape == (0, 64)
