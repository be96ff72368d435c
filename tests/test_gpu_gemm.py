"""GPU parity of the tcgen05 W8A8 scaled product (M > 16) and of the whole
layer (dynamic activation quantization followed by the product) against the
CPU oracle ("[Kernel][FP8] Initial support with dynamic per-tensor scaling",
torch._scaled_mm; "Marlin fp8", per-channel weight scales; "RFC: FP8
Quantization Schema in vLLM", static input scale and output_scale)."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import (DEV, assert_e4m3_close, assert_gemm_close, assert_status_ok, dev, host,
                      sample_rows, scalar, scaled_mm_ref_rows)

pytestmark = pytest.mark.gpu


def _operands(M, N, K, per_channel, seed, outliers=0.0):
    x = synthetic.activation(M, K, torch.bfloat16, seed=seed, outlier_frac=outliers)
    w = synthetic.weight(N, K, torch.bfloat16, seed=seed)
    qa, sa = oracle.quant_per_tensor(x)
    if per_channel:
        qw, sw = oracle.quant_per_row(w)
    else:
        qw, s = oracle.quant_per_tensor(w)
        sw = np.array([s], np.float32)
    return x, w, qa, sa, qw, sw


@pytest.mark.parametrize("out", ["bf16", "fp16", "e4m3"])
@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("M,N,K", [(17, 16, 16), (32, 48, 80), (128, 256, 128), (129, 272, 144),
                                   (200, 512, 512), (300, 784, 1040), (512, 1024, 4096)])
def test_tcgen05_small_shapes(M, N, K, per_channel, out):
    # token x channel tiles at every M (the automatic choice runs the
    # swapped-operand product up to 128 tokens)
    _, _, qa, sa, qw, sw = _operands(M, N, K, per_channel, seed=M * 7 + N * 3 + K)
    y_ref = oracle.scaled_mm_ref(qa, qw, sa, sw)
    if out == "e4m3":
        os_ = np.float32(np.abs(y_ref).max() / 448.0 * 0.8)
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(sa), dev(sw), out_dtype=torch.uint8,
                             out_scale=scalar(os_), kernel="tiled")
        assert_e4m3_close(host(y), y_ref, os_, (M, N, K))
    else:
        dt = torch.bfloat16 if out == "bf16" else torch.float16
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(sa), dev(sw), out_dtype=dt, kernel="tiled")
        assert_gemm_close(host(y), y_ref, (M, N, K, out))
    assert_status_ok()


def test_tcgen05_exact_integer():
    # codes in {-2,-1,-0.5,0,0.5,1,2} and K * 4 < 2^24: the fp32 accumulation
    # is exact, so the output must equal the rounded exact product bit for bit
    codes = np.array([0x40, 0x38, 0x30, 0x00, 0xB0, 0xB8, 0xC0], np.uint8)
    rng = np.random.default_rng(21)
    M, N, K = 257, 384, 2048
    qa = codes[rng.integers(0, 7, (M, K))]
    qw = codes[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.25), dev(sw), out_dtype=torch.bfloat16))
    exact = oracle.scaled_mm_ref(qa, qw, np.float32(0.25), sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    bad = np.argwhere(y != want)
    assert bad.size == 0, (bad[:5], y[tuple(bad[0])], want[tuple(bad[0])])


def test_tcgen05_permutation_weights():
    # W a permutation matrix with distinct power-of-two per-channel scales:
    # y[m, n] = sa * sw[n] * dec(a[m, pi(n)]) exactly; catches any transposed
    # operand, swizzle or column/scale mix-up in the tile pipeline
    K = N = 512
    pi = (np.arange(N) * 101 + 7) % K
    qw = np.zeros((N, K), np.uint8)
    qw[np.arange(N), pi] = 0x38
    rng = np.random.default_rng(3)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    M = 200
    qa = rng.choice(finite, size=(M, K)).astype(np.uint8)
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16))
    want = oracle.decode_table()[qa][:, pi] * 0.5 * sw[None, :]
    want = torch.from_numpy(want).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y, want)


def test_tcgen05_many_tiles_persistent():
    # more tiles than SMs: every CTA loops over several tiles and both TMEM
    # accumulators
    M, N, K = 2048, 4096, 512
    _, _, qa, sa, qw, sw = _operands(M, N, K, True, seed=77)
    y = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(sa), dev(sw), out_dtype=torch.bfloat16)
    yh = host(y)
    rows = sample_rows(M, 96, seed=1)
    assert_gemm_close(yh[rows], scaled_mm_ref_rows(qa[rows], qw, sa, sw))
    assert_status_ok()


def test_tiny_workload_full_path():
    wl = synthetic.WORKLOADS["tiny_w8a8"]
    M, N, K = wl.shapes[0]
    x = synthetic.activation(M, K, torch.bfloat16, seed=wl.seed(0))
    w = synthetic.weight(N, K, torch.bfloat16, seed=wl.seed(0))
    qa, sa = fl.fp8_quant_per_tensor(dev(x))
    qw, sw = fl.fp8_quant_per_tensor(dev(w))
    y = fl.fp8_scaled_mm(qa, qw, sa, sw, out_dtype=torch.bfloat16)
    qa_o, sa_o = oracle.quant_per_tensor(x)
    qw_o, sw_o = oracle.quant_per_tensor(w)
    assert np.array_equal(host(qa), qa_o) and np.array_equal(host(qw), qw_o)
    assert host(sa)[0] == sa_o and host(sw)[0] == sw_o
    # brute force on this small case
    assert_gemm_close(host(y), oracle.scaled_mm_bruteforce(qa_o, qw_o, sa_o, [sw_o]))


def _full_path_sampled(M, N, K, seed, outliers=0.0, rows_count=64, per_channel=False):
    """Dynamic activation quant + product on the GPU; the oracle quantizes the
    same inputs (codes must match bit for bit) and computes sampled rows."""
    x = synthetic.activation(M, K, torch.bfloat16, seed=seed, outlier_frac=outliers)
    w = synthetic.weight(N, K, torch.bfloat16, seed=seed)
    xd, wd = dev(x), dev(w)
    qa, sa = fl.fp8_quant_per_tensor(xd)
    if per_channel:
        qw, sw = fl.fp8_quant_per_row(wd)
    else:
        qw, sw = fl.fp8_quant_per_tensor(wd)
    y = fl.fp8_scaled_mm(qa, qw, sa, sw, out_dtype=torch.bfloat16)
    yh = host(y)
    qa_o, sa_o = oracle.quant_per_tensor(x)
    if per_channel:
        qw_o, sw_o = oracle.quant_per_row(w)
    else:
        qw_o, s = oracle.quant_per_tensor(w)
        sw_o = np.array([s], np.float32)
    assert np.float32(host(sa)[0]) == sa_o
    assert np.array_equal(host(sw).reshape(-1), np.asarray(sw_o).reshape(-1))
    assert np.array_equal(host(qa), qa_o)
    assert np.array_equal(host(qw), qw_o)
    rows = sample_rows(M, rows_count, seed=seed)
    assert_gemm_close(yh[rows], scaled_mm_ref_rows(qa_o[rows], qw_o, sa_o, sw_o), (M, N, K))
    assert_status_ok()


@pytest.mark.parametrize("shape_idx", [0, 1])
def test_prefill_outlier_workload(shape_idx):
    wl = synthetic.WORKLOADS["prefill_w8a8_outliers"]
    M, N, K = wl.shapes[shape_idx]
    _full_path_sampled(M, N, K, wl.seed(shape_idx), outliers=0.01, rows_count=1024)


@pytest.mark.parametrize("nk", [(28672, 4096), (4096, 14336)])
def test_llama8b_largest_m(nk):
    wl = synthetic.WORKLOADS["llama3_8b_w8a8_sweep"]
    idx = wl.shapes.index((8192,) + nk)
    _full_path_sampled(8192, nk[0], nk[1], wl.seed(idx))


@pytest.mark.parametrize("shape", [(128, 6144, 4096), (1024, 4096, 4096)])
def test_llama8b_mid_m(shape):
    wl = synthetic.WORKLOADS["llama3_8b_w8a8_sweep"]
    _full_path_sampled(*shape, wl.seed(wl.shapes.index(shape)), rows_count=shape[0])


@pytest.mark.parametrize("shape", [(64, 10240, 8192), (1024, 8192, 28672), (4096, 57344, 8192)])
def test_llama70b_static_fp8_output(shape):
    """Static input scale from a calibration draw, per-channel weight scale,
    E4M3 output through output_scale (sampled rows)."""
    wl = synthetic.WORKLOADS["llama70b_static_fp8out"]
    M, N, K = shape
    seed = wl.seed(wl.shapes.index(shape))
    rows = sample_rows(M, 48, seed=seed)
    calib = synthetic.activation(256, K, torch.bfloat16, seed=synthetic.calibration_seed(seed))
    x = synthetic.activation(M, K, torch.bfloat16, seed=seed)
    # weights: only the per-row quantization of sampled channels is needed on
    # the CPU; the full matrix goes to the GPU
    w = synthetic.weight(N, K, torch.bfloat16, seed=seed)
    sa_o = oracle.scale_from_amax(oracle.amax(calib))
    qa_o, _ = oracle.quant_per_tensor(x, scale=sa_o)
    qw_o, sw_o = oracle.quant_per_row(w)
    y_cal = scaled_mm_ref_rows(oracle.quant_per_tensor(calib[:32], scale=sa_o)[0], qw_o, sa_o, sw_o)
    os_ = oracle.scale_from_amax(np.float32(np.abs(y_cal).max()))
    qa, _ = fl.fp8_quant_per_tensor(dev(x), scale=scalar(sa_o), dynamic=False)
    qw, sw = fl.fp8_quant_per_row(dev(w))
    y = fl.fp8_scaled_mm(qa, qw, scalar(sa_o), sw, out_dtype=torch.uint8, out_scale=scalar(os_))
    assert np.array_equal(host(qa), qa_o)
    assert np.array_equal(host(sw), sw_o) and np.array_equal(host(qw), qw_o)
    y_ref = scaled_mm_ref_rows(qa_o[rows], qw_o, sa_o, sw_o)
    assert_e4m3_close(host(y)[rows], y_ref, os_, shape)
    assert_status_ok()


def test_zero_rows_launch_nothing():
    qa = torch.zeros((0, 64), dtype=torch.uint8, device=DEV)
    qw = torch.zeros((32, 64), dtype=torch.uint8, device=DEV)
    y = fl.fp8_scaled_mm(qa, qw, scalar(1.0), scalar(1.0))
    assert y.shape == (0, 32)


@pytest.mark.parametrize("M,N,K", [(100, 512, 4096), (64, 4096, 4096), (128, 768, 1152)])
def test_tcgen05_split_k_exact_integer(M, N, K):
    # few output tiles: CTAs of a cluster split K and add their fp32 partial
    # tiles through distributed shared memory; with exact-integer operands
    # every partial and the total are exact, so the result is bit-exact
    codes = np.array([0x40, 0x38, 0x30, 0x00, 0xB0, 0xB8, 0xC0], np.uint8)
    rng = np.random.default_rng(M + N + K)
    qa = codes[rng.integers(0, 7, (M, K))]
    qw = codes[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16,
                              kernel="tiled"))
    exact = oracle.scaled_mm_ref(qa, qw, np.float32(0.5), sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y, want)
    assert_status_ok()


@pytest.mark.parametrize("M,N,K", [(1024, 4096, 512), (1024, 11008, 256), (1000, 10240, 384),
                                   (1024, 4112, 256), (1024, 57344, 128)])
def test_tcgen05_prefill_shapes_exact_integer(M, N, K):
    # persistent launches over the prefill and 70B widths, one with a
    # 16-column tail in its last 256-column tile (N = 4112) and one with an M
    # tail (M = 1000); exact-integer operands make the result bit-exact
    codes = np.array([0x40, 0x38, 0x30, 0x00, 0xB0, 0xB8, 0xC0], np.uint8)
    rng = np.random.default_rng(M + 3 * N + K)
    qa = codes[rng.integers(0, 7, (M, K))]
    qw = codes[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16))
    exact = oracle.scaled_mm_ref(qa, qw, np.float32(0.5), sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y, want)
    assert_status_ok()
