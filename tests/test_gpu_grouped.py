"""GPU parity of the grouped W8A8 product for mixture-of-experts layers
(fp8_grouped_mm; "RFC: FP8 Quantization Schema in vLLM", the gate_proj
question) against the CPU oracle's grouped product: expert e takes rows
offsets[e] .. offsets[e+1]-1, with offsets in device memory."""
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
FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)


def _offsets(sizes, start=0):
    return np.concatenate([[start], start + np.cumsum(sizes)]).astype(np.int32)


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("per_token", [False, True])
def test_exact_integer_ragged_groups(per_channel, per_token):
    # group sizes 0, 1, 127, 128, 129, 300 and more; rows before the first
    # and after the last group stay untouched; exact fp32 accumulation, so
    # the output must be the rounded exact product bit for bit
    rng = np.random.default_rng(1 + 2 * per_channel + per_token)
    sizes = [0, 1, 127, 128, 129, 300, 5, 0, 40]
    E, N, K = len(sizes), 272, 512
    offs = _offsets(sizes, start=3)
    M = int(offs[-1]) + 6
    qa = CODES[rng.integers(0, 7, (M, K))]
    qw = CODES[rng.integers(0, 7, (E, N, K))]
    sw = (np.array([[2.0 ** ((n + e) % 7 - 3) for n in range(N)] for e in range(E)], np.float32)
          if per_channel else np.array([2.0 ** (e % 5 - 2) for e in range(E)], np.float32))
    sa = (np.array([2.0 ** (m % 5 - 2) for m in range(M)], np.float32) if per_token
          else np.array([0.75], np.float32))
    y0 = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    y = fl.fp8_grouped_mm(dev(qa), dev(qw), dev(offs), dev(sa), dev(sw), y=y0,
                          per_token=per_token)
    yh = host(y)
    exact = oracle.grouped_mm_bruteforce(qa, qw, offs, sa, sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    lo, hi = offs[0], offs[-1]
    assert np.all(yh[:lo] == 7.0) and np.all(yh[hi:] == 7.0)
    bad = np.argwhere(yh[lo:hi] != want[lo:hi])
    assert bad.size == 0, (bad[:5],)
    assert_status_ok()


@pytest.mark.parametrize("out", ["bf16", "e4m3"])
def test_mixture_of_experts_layer(out):
    # 8 experts, 2048 tokens routed top-2 (4096 rows, uneven expert loads),
    # expert weights quantized per channel, activations per tensor
    E, N, K = 8, 2048, 1024
    rng = np.random.default_rng(8)
    load = rng.dirichlet(np.ones(E) * 0.7)
    sizes = np.floor(load * 4096).astype(int)
    sizes[-1] += 4096 - sizes.sum()
    offs = _offsets(sizes)
    M = int(offs[-1])
    x = synthetic.activation(M, K, torch.bfloat16, seed=21)
    qa, sa = fl.fp8_quant_per_tensor(dev(x))
    qw_list, sw_list = [], []
    for e in range(E):
        q, s = oracle.quant_per_row(synthetic.weight(N, K, torch.bfloat16, seed=100 + e))
        qw_list.append(q)
        sw_list.append(s)
    qw, sw = np.stack(qw_list), np.stack(sw_list)
    qa_h, sa_h = host(qa), host(sa)[0]
    rows = sample_rows(M, 96, seed=2)
    y_ref = oracle.grouped_mm_ref(qa_h, qw, offs, sa_h, sw)[rows]
    if out == "e4m3":
        os_ = np.float32(np.abs(y_ref).max() / 448.0 * 0.8)
        y = fl.fp8_grouped_mm(qa, dev(qw), dev(offs), sa, dev(sw), out_dtype=torch.uint8,
                              out_scale=scalar(os_))
        assert_e4m3_close(host(y)[rows], y_ref, os_)
    else:
        y = fl.fp8_grouped_mm(qa, dev(qw), dev(offs), sa, dev(sw))
        assert_gemm_close(host(y)[rows], y_ref)
    assert_status_ok()


def test_decode_sized_groups_many_experts():
    # 64 experts with 0..6 tokens each: every tile is mostly padding rows
    E, N, K = 64, 512, 2048
    rng = np.random.default_rng(64)
    sizes = rng.integers(0, 7, E)
    offs = _offsets(sizes)
    M = int(offs[-1])
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qw = rng.choice(FINITE, size=(E, N, K)).astype(np.uint8)
    sw = rng.uniform(1e-3, 2e-3, E).astype(np.float32)
    y = fl.fp8_grouped_mm(dev(qa), dev(qw), dev(offs), scalar(0.01), dev(sw))
    assert_gemm_close(host(y), oracle.grouped_mm_ref(qa, qw, offs, np.float32(0.01), sw))


def test_offsets_change_between_graph_replays():
    # the routing (device offsets) changes between replays of one captured
    # graph: the product follows without a new capture
    E, N, K, M = 4, 256, 256, 200
    rng = np.random.default_rng(9)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qw = rng.choice(FINITE, size=(E, N, K)).astype(np.uint8)
    sw = np.full(E, 1e-3, np.float32)
    offs_d = dev(_offsets([50, 50, 50, 50]))
    a_d, w_d, sa_d, sw_d = dev(qa), dev(qw), scalar(0.02), dev(sw)
    y = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    ws = fl.workspace(DEV)
    fl.fp8_grouped_mm(a_d, w_d, offs_d, sa_d, sw_d, y=y, ws=ws)  # set-up outside capture
    s = torch.cuda.Stream(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fl.fp8_grouped_mm(a_d, w_d, offs_d, sa_d, sw_d, y=y, ws=ws)
    for sizes in ([50, 50, 50, 50], [0, 200, 0, 0], [7, 129, 1, 63]):
        offs = _offsets(sizes)
        offs_d.copy_(torch.from_numpy(offs))
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_gemm_close(host(y), oracle.grouped_mm_ref(qa, qw, offs, np.float32(0.02), sw))


def test_gate_padded_to_16_channels():
    # an 8-expert gate: weights padded with 8 zero rows to N = 16 (the FP8
    # shape rule); the first 8 logits match the oracle, the rest are 0
    M, K = 64, 1024
    rng = np.random.default_rng(10)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    gate = rng.choice(FINITE, size=(8, K)).astype(np.uint8)
    padded = np.concatenate([gate, np.zeros((8, K), np.uint8)])
    y = host(fl.fp8_scaled_mm(dev(qa), dev(padded), scalar(0.01), scalar(0.02),
                              out_dtype=torch.float16))
    assert np.all(y[:, 8:] == 0)
    assert_gemm_close(y[:, :8], oracle.scaled_mm_ref(qa, gate, np.float32(0.01),
                                                     [np.float32(0.02)]))
