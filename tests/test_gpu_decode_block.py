"""The Llama-3-8B-shaped decode layer chained through the library and
captured in one CUDA graph ("Marlin fp8": FP8 decode pays off with CUDA
graphs); at one token the W8A8 layer's o, gate/up and down products run with
their quantization fused.  Each stage is compared with the CPU oracle on the input the GPU
gave it, and graph replays must reproduce eager execution bit for bit."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from fp8_quantized_linear_gb300.block import ORDER, SHAPES, DecodeBlock
from gpu_util import DEV, assert_gemm_close, assert_status_ok, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def weights():
    return {name: synthetic.weight(N, K, torch.bfloat16, seed=300 + i)
            for i, (name, (N, K)) in enumerate(SHAPES.items())}


def _block(M, kind, weights, seed):
    wd = {k: v.to(DEV) for k, v in weights.items()}
    gamma = synthetic.norm_weight(4096, torch.bfloat16, seed=seed).to(DEV)
    blk = DecodeBlock(M, wd, kind=kind, gamma=gamma)
    x = synthetic.activation(M, 4096, blk.act_dtype, seed=seed)
    blk.x.copy_(x.to(DEV))
    return blk, x


@pytest.mark.parametrize("kind", ["w8a16", "w8a8"])
@pytest.mark.parametrize("M", [1, 16])
def test_stages_against_oracle(M, kind, weights):
    blk, x = _block(M, kind, weights, seed=M)
    blk.forward()
    torch.cuda.synchronize()
    for name in ORDER:
        qw, sw = oracle.quant_per_row(weights[name])
        inp = blk.input_of(name)
        if kind == "w8a16":
            y_ref = oracle.w8a16_ref(inp.cpu(), qw, sw)
        else:
            if name == "qkv":
                _, _, h = fl.fp8_rmsnorm_quant(blk.x, blk.gamma, blk.eps, want_h=True)
                src = host(h)
            else:
                src = host(inp)
            q_o, s_o = oracle.quant_per_tensor(src.astype(np.float32))
            if not blk.fused(name):  # a fused product never writes its codes
                assert np.array_equal(host(blk.qa[name]), q_o), name
            assert np.float32(host(blk.sa[name])[0]) == s_o, name
            y_ref = oracle.scaled_mm_ref(q_o, qw, s_o, sw)
        assert_gemm_close(host(blk.y[name]), y_ref, (kind, M, name))
    if kind == "w8a8":
        assert_status_ok()


@pytest.mark.parametrize("kind", ["w8a16", "w8a8"])
def test_graph_replay_equals_eager(kind, weights):
    M = 4
    blk, _ = _block(M, kind, weights, seed=11)
    blk.capture()
    for seed in (12, 13):
        x = synthetic.activation(M, 4096, blk.act_dtype, seed=seed).to(DEV)
        blk.x.copy_(x)
        blk.forward()
        torch.cuda.synchronize()
        eager = {name: blk.y[name].clone() for name in ORDER}
        for name in ORDER:
            blk.y[name].zero_()
        blk.graph.replay()
        torch.cuda.synchronize()
        for name in ORDER:
            assert torch.equal(blk.y[name], eager[name]), (kind, seed, name)
