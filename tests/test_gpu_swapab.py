"""GPU parity of the swapped-operand tcgen05 product (FP8L_KERNEL_SWAPPED):
128 weight rows by M <= 128 tokens per tile, with clusters splitting K when
the weight blocks are fewer than the CTA slots.  Against the CPU oracle:
exact-integer products bit for bit (ragged N and K tails, K below one
k-block, every split size the launcher picks), permutation weights exactly,
Gaussian operands within the layer's tolerance for every scale and output
form, the full-size few-token shapes on sampled rows, and the same products
through the other two kernels."""
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
FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)


def _exact_case(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qa = CODES[rng.integers(0, 7, (M, K))]
    qw = CODES[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    return qa, qw, sw


# N = 16: one partial weight block (split up to 8); 2320: ragged last block;
# 4096 and 6144: split 8 and 6; 28672: no split.  K = 16 and 96: one partial
# k-block; 640: five; 4096: thirty-two.
@pytest.mark.parametrize("M", [1, 5, 16, 17, 64, 100, 128])
@pytest.mark.parametrize("N,K", [(16, 96), (2320, 640), (4096, 4096), (6144, 16), (28672, 640)])
def test_exact_integer(M, N, K):
    qa, qw, sw = _exact_case(M, N, K, seed=M * 7 + N + K)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16,
                              kernel="swapped"))
    exact = scaled_mm_ref_rows(qa, qw, np.float32(0.5), sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    bad = np.argwhere(y != want)
    assert bad.size == 0, (bad[:5],)
    assert_status_ok()


@pytest.mark.parametrize("stable", [False, True])
@pytest.mark.parametrize("M", [3, 48])
def test_permutation_weights(M, stable):
    K = N = 1024
    pi = (np.arange(N) * 389 + 11) % K
    qw = np.zeros((N, K), np.uint8)
    qw[np.arange(N), pi] = 0x38
    rng = np.random.default_rng(16 + M)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16,
                              kernel="swapped", stable_weights=stable))
    want = oracle.decode_table()[qa][:, pi] * 0.5 * sw[None, :]
    want = torch.from_numpy(want).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y, want)


@pytest.mark.parametrize("out", ["bf16", "fp16", "e4m3"])
@pytest.mark.parametrize("per_token", [False, True])
@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("M", [1, 16, 80])
def test_gaussian_operands(M, out, per_token, per_channel):
    N, K = 6144, 4096
    x = synthetic.activation(M, K, torch.bfloat16, seed=177 + M, outlier_frac=0.01)
    w = synthetic.weight(N, K, torch.bfloat16, seed=177)
    qa, sa = (oracle.quant_per_row(x) if per_token else oracle.quant_per_tensor(x))
    qw, sw = oracle.quant_per_row(w) if per_channel else oracle.quant_per_tensor(w)
    sw = np.atleast_1d(np.asarray(sw, np.float32))
    y_ref = scaled_mm_ref_rows(qa, qw, sa, sw)
    sa_d = dev(np.atleast_1d(np.asarray(sa, np.float32)))
    if out == "e4m3":
        os_ = np.float32(np.abs(y_ref).max() / 448.0 * 0.8)
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), sa_d, dev(sw), out_dtype=torch.uint8,
                             out_scale=scalar(os_), per_token=per_token, kernel="swapped")
        assert_e4m3_close(host(y), y_ref, os_)
    else:
        dt = torch.bfloat16 if out == "bf16" else torch.float16
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), sa_d, dev(sw), out_dtype=dt, per_token=per_token,
                             kernel="swapped")
        assert_gemm_close(host(y), y_ref)
    assert_status_ok()


# the few-token shapes of the Llama-3-8B and 70B sets at full size: W8A8
# with per-tensor scales and bf16 out, and static scales with per-channel
# weight scales and E4M3 out; sampled rows against the oracle
@pytest.mark.parametrize("M,N,K,e4m3", [(16, 28672, 4096, False), (128, 4096, 14336, False),
                                        (1, 57344, 8192, True), (64, 10240, 8192, True)])
def test_full_size_shapes(M, N, K, e4m3):
    x = synthetic.activation(M, K, torch.bfloat16, seed=M + N)
    w = synthetic.weight(N, K, torch.bfloat16, seed=N + K)
    qa, sa = oracle.quant_per_tensor(x)
    qw, sw = oracle.quant_per_row(w) if e4m3 else oracle.quant_per_tensor(w)
    sw = np.atleast_1d(np.asarray(sw, np.float32))
    rows = sample_rows(M, 8, seed=5)
    y_ref = scaled_mm_ref_rows(qa[rows], qw, sa, sw)
    if e4m3:
        os_ = np.float32(np.abs(y_ref).max() / 448.0 * 0.8)
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(sa), dev(sw), out_dtype=torch.uint8,
                             out_scale=scalar(os_), kernel="swapped", stable_weights=True)
        assert_e4m3_close(host(y)[rows], y_ref, os_)
    else:
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(sa), dev(sw), out_dtype=torch.bfloat16,
                             kernel="swapped", stable_weights=True)
        assert_gemm_close(host(y)[rows], y_ref)
    assert_status_ok()


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_all_kernels_agree_on_exact_products(M):
    # exact-integer operands: every kernel's result is the exact value rounded
    # once, so all three agree bit for bit
    N, K = 3072, 2048
    qa, qw, sw = _exact_case(M, N, K, seed=400 + M)
    a, w, s1, s2 = dev(qa), dev(qw), scalar(0.25), dev(sw)
    ys = {k: host(fl.fp8_scaled_mm(a, w, s1, s2, out_dtype=torch.float16, kernel=k))
          for k in ("stream", "swapped", "tiled")}
    assert np.array_equal(ys["swapped"], ys["stream"])
    assert np.array_equal(ys["swapped"], ys["tiled"])


def test_graph_replay_with_stable_weights():
    # a chain of few-token products captured in one CUDA graph, each launched
    # as a programmatic dependent that loads weights before its wait; the
    # second product reads the first one's output
    M, N, K = 16, 4096, 4096
    x = synthetic.activation(M, K, torch.bfloat16, seed=31)
    w1 = synthetic.weight(N, K, torch.bfloat16, seed=32)
    w2 = synthetic.weight(K, N, torch.bfloat16, seed=33)
    qa, sa = oracle.quant_per_tensor(x)
    qw1, sw1 = oracle.quant_per_tensor(w1)
    qw2, sw2 = oracle.quant_per_tensor(w2)
    y1_ref = scaled_mm_ref_rows(qa, qw1, sa, [sw1])
    os1 = np.float32(np.abs(y1_ref).max() / 448.0)
    a, b1, b2 = dev(qa), dev(qw1), dev(qw2)
    s_a, s_1, s_2, s_o = scalar(sa), scalar(sw1), scalar(sw2), scalar(os1)
    y1 = torch.empty((M, N), dtype=torch.uint8, device=a.device)
    y2 = torch.empty((M, K), dtype=torch.bfloat16, device=a.device)
    ws = fl.workspace(a.device)
    stream = torch.cuda.Stream(a.device)

    def step():
        fl.fp8_scaled_mm(a, b1, s_a, s_1, out_dtype=torch.uint8, out_scale=s_o, y=y1, ws=ws,
                         kernel="swapped", stable_weights=True)
        fl.fp8_scaled_mm(y1, b2, s_o, s_2, out_dtype=torch.bfloat16, y=y2, ws=ws,
                         kernel="swapped", stable_weights=True)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    y1.zero_()
    y2.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    q1 = host(y1).astype(np.uint8)
    assert_e4m3_close(q1, y1_ref, os1)
    y2_ref = scaled_mm_ref_rows(q1, qw2, os1, [sw2])
    assert_gemm_close(host(y2), y2_ref)
    assert_status_ok()


def test_m_above_128_is_refused():
    a = torch.zeros((129, 64), dtype=torch.uint8, device="cuda")
    w = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError):
        fl.fp8_scaled_mm(a, w, scalar(1.0), scalar(1.0), kernel="swapped")
