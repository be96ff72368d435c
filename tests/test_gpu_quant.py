"""GPU parity of the per-tensor / per-row E4M3 quantizer: codes and scales
must equal the oracle's bit for bit ("[Kernel][FP8] Initial support with
dynamic per-tensor scaling", Algorithm; "RFC: FP8 Quantization Schema in
vLLM", static input scale)."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import pins
import synthetic
from gpu_util import DEV, assert_status_ok, dev, host, scalar

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float16, torch.float32]


def _check_dynamic(x):
    q, s = fl.fp8_quant_per_tensor(dev(x))
    q_o, s_o = oracle.quant_per_tensor(x)
    qh = host(q)
    assert np.float32(host(s)[0]) == s_o, (host(s)[0], s_o)
    bad = np.nonzero(qh.reshape(-1) != q_o.reshape(-1))[0]
    assert bad.size == 0, (x.dtype, tuple(x.shape), bad[:8], qh.reshape(-1)[bad[:8]], q_o.reshape(-1)[bad[:8]])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 1), (1, 15), (1, 16), (1, 17), (3, 33), (16, 512),
                                   (37, 1000), (129, 4112), (1024, 4096)])
def test_dynamic_matches_oracle(dtype, shape):
    x = synthetic.activation(shape[0], shape[1], dtype, seed=shape[0] * 131 + shape[1])
    _check_dynamic(x)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_dynamic_outlier_channels(dtype):
    # prefill workload: 1% of K channels scaled by 50 (many small codes,
    # E4M3 subnormals)
    x = synthetic.activation(1024, 4096, dtype, seed=3000, outlier_frac=0.01)
    _check_dynamic(x)


def test_dynamic_llama_sizes():
    for (M, K) in ((8192, 4096), (8192, 14336)):
        _check_dynamic(synthetic.activation(M, K, torch.bfloat16, seed=M + K))


def test_empty_and_zero():
    x = torch.zeros((0, 64), dtype=torch.bfloat16)
    q, s = fl.fp8_quant_per_tensor(dev(x))
    assert host(s)[0] == 1.0 and q.numel() == 0
    x = torch.zeros((5, 48), dtype=torch.float16)
    q, s = fl.fp8_quant_per_tensor(dev(x))
    assert host(s)[0] == 1.0 and not host(q).any()
    x = -torch.zeros((2, 16), dtype=torch.float32)  # negative zeros keep their sign
    _check_dynamic(x)


def test_worked_examples():
    def quant(x, scale=None):
        q, s = fl.fp8_quant_per_tensor(dev(x.reshape(1, -1)))
        return host(q).reshape(-1), np.float32(host(s)[0])
    pins.check_quant_worked(quant)


def test_single_huge_element_and_ties():
    # amax set by one element; every other element sits on an E4M3 tie after
    # division by s = 2^-6
    table = oracle.decode_table()
    pos = table[:127]
    mids = ((pos[:-1] + pos[1:]) / 2) / 64.0
    vals = np.concatenate([[7.0], mids, -mids]).astype(np.float32)
    _check_dynamic(torch.from_numpy(vals).reshape(1, -1))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.0517578125e-05, 7.0])
def test_static_every_16bit_value(dtype, scale):
    # every finite value of the format, static scale: exhaustive cast check
    v = torch.from_numpy(pins.all_16bit_values(dtype)).to(dtype)
    x = v.reshape(1, -1)
    q, _ = fl.fp8_quant_per_tensor(dev(x), scale=scalar(scale), dynamic=False)
    q_o, _ = oracle.quant_per_tensor(x, scale=np.float32(scale))
    assert np.array_equal(host(q).reshape(-1), q_o.reshape(-1))


def _many_scales():
    """The fast-path limits of the kernels' quotient (2^-92 and 2^100) and
    their float32 neighbours on both sides, other landmarks (subnormal and
    huge scales, reciprocals that are not exact), and 256 seeded scales with
    random significands and exponents in [-100, 100]."""
    f32 = np.float32
    lims = [f32(2.0 ** -92), f32(2.0 ** 100)]
    out = []
    for v in lims:
        out += [np.nextafter(v, f32(0)), v, np.nextafter(v, f32(np.inf))]
    out += [f32(2.0 ** -93), f32(2.0 ** 101), f32(2.0 ** -126), f32(1e-40), f32(3e38),
            f32(1.0), f32(0.1), f32(1.0 / 3.0), f32(7.0), f32(1.0 / 448.0), f32(2.0 ** -9),
            f32(448.0)]
    rng = np.random.default_rng(2024)
    sig = rng.integers(0, 1 << 23, 256, dtype=np.uint32)
    exp = rng.integers(-100, 101, 256)
    out += list(((((127 + exp) << 23).astype(np.uint32)) | sig).view(np.float32))
    return [f32(v) for v in out]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_static_every_16bit_value_many_scales(dtype):
    # every finite value of the format under 274 scales: the kernels' codes
    # (corrected quotient, or IEEE division outside [2^-92, 2^100]) against
    # the oracle's IEEE division, bit for bit
    v = torch.from_numpy(pins.all_16bit_values(dtype)).to(dtype)
    x = v.reshape(1, -1)
    xd = dev(x)
    for s in _many_scales():
        q, _ = fl.fp8_quant_per_tensor(xd, scale=scalar(s), dynamic=False)
        q_o, _ = oracle.quant_per_tensor(x, scale=s)
        assert np.array_equal(host(q).reshape(-1), q_o.reshape(-1)), (dtype, float(s))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_dynamic_every_16bit_value_below_an_amax(dtype):
    # dynamic mode: the finite values of the format up to a chosen maximum A
    # (both signs), for 48 maxima of various exponents and significands; the
    # scale RN(A / 448) and every code must equal the oracle's
    v = pins.all_16bit_values(dtype)
    pos = np.unique(np.abs(v[np.isfinite(v)]))
    rng = np.random.default_rng(7)
    picks = np.concatenate([pos[-1:], pos[rng.integers(len(pos) // 4, len(pos) - 1, 47)]])
    for a in picks:
        sel = v[np.abs(v) <= a]
        x = torch.from_numpy(sel).to(dtype).reshape(1, -1)
        q, s = fl.fp8_quant_per_tensor(dev(x))
        q_o, s_o = oracle.quant_per_tensor(x)
        assert np.float32(host(s)[0]) == s_o, (dtype, float(a))
        assert np.array_equal(host(q).reshape(-1), q_o.reshape(-1)), (dtype, float(a))


def test_static_float32_midpoint_neighbourhoods():
    # every E4M3 rounding midpoint and 64 float32 neighbours on each side
    table = oracle.decode_table()
    pos = table[:127]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    mids = np.concatenate([mids, np.float32([448.0, 464.0, 480.0, 1e6])])
    bits = mids.view(np.int32)
    offs = np.arange(-64, 65, dtype=np.int32)
    v = (bits[:, None] + offs[None, :]).reshape(-1).view(np.float32)
    v = np.concatenate([v, -v])
    x = torch.from_numpy(v).reshape(1, -1)
    for scale in (1.0, 0.5, 0.1, 1e-3):
        q, _ = fl.fp8_quant_per_tensor(dev(x), scale=scalar(scale), dynamic=False)
        q_o, _ = oracle.quant_per_tensor(x, scale=np.float32(scale))
        assert np.array_equal(host(q).reshape(-1), q_o.reshape(-1)), scale


def test_static_random_float32():
    g = torch.Generator().manual_seed(77)
    x = (torch.randn(1 << 20, generator=g) * torch.exp2(torch.randint(-30, 20, (1 << 20,), generator=g).float()))
    for scale in (1.0, 0.37, 2.5e-4):
        q, _ = fl.fp8_quant_per_tensor(dev(x.reshape(64, -1)), scale=scalar(scale), dynamic=False)
        q_o, _ = oracle.quant_per_tensor(x, scale=np.float32(scale))
        assert np.array_equal(host(q).reshape(-1), q_o.reshape(-1)), scale


def test_repeat_and_workspace_reuse():
    # stale partials from a larger earlier call must not leak into a smaller one
    big = synthetic.activation(4096, 4096, torch.bfloat16, seed=5) * 10
    small = synthetic.activation(4, 64, torch.bfloat16, seed=6)
    fl.fp8_quant_per_tensor(dev(big))
    _check_dynamic(small)
    q1, s1 = fl.fp8_quant_per_tensor(dev(small))
    q2, s2 = fl.fp8_quant_per_tensor(dev(small))
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    assert_status_ok()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 16), (7, 48), (256, 512), (300, 4096)])
def test_per_row_matches_oracle(dtype, shape):
    w = synthetic.weight(shape[0], shape[1], dtype, seed=shape[0] + 7 * shape[1])
    if shape[0] > 3:
        w[3] = 0  # an all-zero row gets scale 1
    q, s = fl.fp8_quant_per_row(dev(w))
    q_o, s_o = oracle.quant_per_row(w)
    assert np.array_equal(host(s), s_o)
    assert np.array_equal(host(q), q_o)


def test_per_row_large():
    w = synthetic.weight(8192, 8192, torch.bfloat16, seed=11)
    q, s = fl.fp8_quant_per_row(dev(w))
    q_o, s_o = oracle.quant_per_row(w)
    assert np.array_equal(host(s), s_o)
    assert np.array_equal(host(q), q_o)


@pytest.mark.parametrize("shape", [(1024, 4096), (8192, 4096)])
def test_dynamic_inside_cuda_graph(shape):
    # the single-pass quantizer is a cooperative launch: it must capture into
    # a CUDA graph and give the oracle's bytes on every replay
    M, K = shape
    x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = fl.workspace(DEV)
    x.copy_(synthetic.activation(M, K, torch.bfloat16, seed=1).to(DEV))
    fl.fp8_quant_per_tensor(x, q=q, scale=s, ws=ws)  # eager first call (set-up)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fl.fp8_quant_per_tensor(x, q=q, scale=s, ws=ws)
    for seed in (2, 3):
        xs = synthetic.activation(M, K, torch.bfloat16, seed=seed, outlier_frac=0.01)
        x.copy_(xs.to(DEV))
        g.replay()
        torch.cuda.synchronize()
        q_o, s_o = oracle.quant_per_tensor(xs)
        assert host(s)[0] == s_o
        assert np.array_equal(host(q), q_o)
    assert_status_ok()


def test_static_streamed_large():
    # static scale on a tensor far larger than the on-chip stages: every
    # piece is streamed once through the ring
    x = synthetic.activation(8192, 4096, torch.bfloat16, seed=21)
    q, _ = fl.fp8_quant_per_tensor(dev(x), scale=scalar(0.0371), dynamic=False)
    q_o, _ = oracle.quant_per_tensor(x, scale=np.float32(0.0371))
    assert np.array_equal(host(q), q_o)


def test_dynamic_float32_streamed():
    # 64 MB of fp32: pass 2 casts the resident pieces and re-reads the rest
    _check_dynamic(synthetic.activation(4096, 4096, torch.float32, seed=22))


@pytest.mark.parametrize("extra_words", [-1, 0, 1, 2049])
def test_dynamic_resident_boundary(extra_words):
    # one block per SM keeps 6 pieces of 2048 16-byte words on chip; these
    # sizes put each block's run just under, at, and just over that
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    n_words = sms * (6 * 2048 + extra_words)
    numel = n_words * 8 + 5  # bf16: 8 elements per word, plus a ragged tail
    x = synthetic.activation(1, numel, torch.bfloat16, seed=23 + extra_words)
    _check_dynamic(x)


def test_alternating_grid_sizes_share_the_workspace():
    # the barrier words alternate between calls; calls with 1 block and with
    # one block per SM interleave on one workspace
    ws = fl.workspace(DEV)
    shapes = [(1, 16), (1024, 4096), (3, 33), (129, 4112), (1, 16), (2048, 4096), (16, 512)]
    for rep in range(2):
        for i, (M, K) in enumerate(shapes):
            x = synthetic.activation(M, K, torch.bfloat16, seed=900 + 10 * rep + i)
            q, s = fl.fp8_quant_per_tensor(dev(x), ws=ws)
            q_o, s_o = oracle.quant_per_tensor(x)
            assert host(s)[0] == s_o, (M, K)
            assert np.array_equal(host(q), q_o), (M, K)
    assert_status_ok()
