"""GPU parity of the weight-streaming kernels: W8A16 ("Marlin fp8": 16-bit
activations, E4M3 weights, one scale per output channel) and the small-M
branch of the W8A8 scaled product."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import DEV, assert_e4m3_close, assert_gemm_close, assert_status_ok, dev, host, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_wait_gave_up():
    # no bounded device-side wait of the calls made with the workspace gave up
    yield
    assert_status_ok()


def _w8a16_case(M, N, K, xdtype, seed, kernel="stream"):
    x = synthetic.activation(M, K, xdtype, seed=seed)
    w = synthetic.weight(N, K, torch.bfloat16, seed=seed)
    qw, sw = oracle.quant_per_row(w)
    y = fl.fp8_w8a16_mm(dev(x), dev(qw), dev(sw), kernel=kernel)
    assert y.dtype == xdtype
    return host(y), oracle.w8a16_ref(x, qw, sw)


@pytest.mark.parametrize("xdtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (1, 32, 80), (3, 48, 208), (8, 256, 512),
                                   (9, 64, 1024), (16, 272, 4096), (17, 64, 256), (40, 80, 144)])
def test_w8a16_small(M, N, K, xdtype):
    y, y_ref = _w8a16_case(M, N, K, xdtype, seed=M * 1000 + N + K)
    assert_gemm_close(y, y_ref, (M, N, K, xdtype))


@pytest.mark.parametrize("shape_idx", range(12))
@pytest.mark.parametrize("kernel", ["stream", "auto"])
def test_w8a16_decode_workload(shape_idx, kernel):
    wl = synthetic.WORKLOADS["decode_w8a16"]
    M, N, K = wl.shapes[shape_idx]
    y, y_ref = _w8a16_case(M, N, K, torch.float16, seed=wl.seed(shape_idx), kernel=kernel)
    assert_gemm_close(y, y_ref, (M, N, K))


def test_w8a16_exact_integer_and_distinct_channel_scales():
    # all-ones weights, integer activations, power-of-two per-channel scales:
    # fp32 accumulation is exact, so each output equals the closed form
    # sw[n] * sum_k x[m,k] exactly (a scale applied to the wrong column, the
    # bug of a kernel that only worked with a repeated scalar scale, fails)
    M, N, K = 5, 64, 512
    g = torch.Generator().manual_seed(4)
    x = torch.randint(-3, 4, (M, K), generator=g).to(torch.float16)
    qw = np.full((N, K), 0x38, np.uint8)
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    y = host(fl.fp8_w8a16_mm(dev(x), dev(qw), dev(sw)))
    want = x.double().sum(1, keepdim=True).numpy() * sw[None, :].astype(np.float64)
    assert np.array_equal(y, want)


@pytest.mark.parametrize("M,K", [(7, 256), (7, 208), (13, 256), (1, 1024), (8, 4096)])
def test_w8a16_permutation_weights(M, K):
    # W is a permutation matrix: y[m, n] = sw[n] * x[m, pi(n)] exactly, so a
    # k position paired with the wrong weight byte anywhere in a chunk fails
    # (K = 208: a ragged last chunk; 13 tokens: two token tiles).
    N = K
    pi = (np.arange(N) * 37 + 11) % K
    qw = np.zeros((N, K), np.uint8)
    qw[np.arange(N), pi] = 0x38
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    x = synthetic.activation(M, K, torch.float16, seed=9 + M + K)
    y = host(fl.fp8_w8a16_mm(dev(x), dev(qw), dev(sw)))
    want = x.double().numpy()[:, pi] * sw[None, :]
    assert np.array_equal(y, want.astype(np.float16).astype(np.float32))


@pytest.mark.parametrize("xdtype", [torch.float16, torch.bfloat16])
def test_w8a16_activations_16_byte_aligned_only(xdtype):
    # activations starting 16 bytes past a 32-byte boundary (the API asks
    # for 16-byte alignment only)
    M, N, K = 4, 256, 1024
    x = synthetic.activation(M, K, xdtype, seed=31)
    w = synthetic.weight(N, K, torch.bfloat16, seed=31)
    qw, sw = oracle.quant_per_row(w)
    buf = torch.empty(M * K + 8, dtype=xdtype, device=DEV)
    xd = buf[8:].view(M, K)
    xd.copy_(dev(x))
    assert xd.data_ptr() % 32 == 16
    y = host(fl.fp8_w8a16_mm(xd, dev(qw), dev(sw)))
    assert_gemm_close(y, oracle.w8a16_ref(x, qw, sw), (M, N, K, xdtype))


def test_w8a16_empty_batch():
    x = torch.zeros((0, 64), dtype=torch.float16)
    qw = np.zeros((32, 64), np.uint8)
    y = fl.fp8_w8a16_mm(dev(x), dev(qw), dev(np.ones(32, np.float32)))
    assert y.shape == (0, 32)


def _w8a8_small(M, N, K, per_channel, out, seed, kernel):
    x = synthetic.activation(M, K, torch.bfloat16, seed=seed)
    w = synthetic.weight(N, K, torch.bfloat16, seed=seed)
    qa, sa = oracle.quant_per_tensor(x)
    if per_channel:
        qw, sw = oracle.quant_per_row(w)
    else:
        qw, s = oracle.quant_per_tensor(w)
        sw = np.array([s], np.float32)
    y_ref = oracle.scaled_mm_ref(qa, qw, sa, sw)
    if out == "e4m3":
        os_ = np.float32(np.abs(y_ref).max() / 448.0 * 0.75)  # a few outputs saturate
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(sa), dev(sw), out_dtype=torch.uint8,
                             out_scale=scalar(os_), kernel=kernel)
        assert_e4m3_close(host(y), y_ref, os_, (M, N, K))
    else:
        dt = torch.bfloat16 if out == "bf16" else torch.float16
        y = fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(sa), dev(sw), out_dtype=dt, kernel=kernel)
        assert_gemm_close(host(y), y_ref, (M, N, K, out))


# the CUDA-core weight-streaming kernel, and the swapped-operand tcgen05
# product the automatic choice takes for most of these shapes
@pytest.mark.parametrize("kernel", ["stream", "swapped"])
@pytest.mark.parametrize("out", ["bf16", "fp16", "e4m3"])
@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (1, 256, 512), (5, 48, 80), (16, 256, 512),
                                   (16, 4096, 4096), (1, 28672, 4096), (16, 4096, 14336)])
def test_w8a8_small_m(M, N, K, per_channel, out, kernel):
    _w8a8_small(M, N, K, per_channel, out, seed=M + N + K, kernel=kernel)


@pytest.mark.parametrize("M,K", [(16, 1024), (8, 1024), (3, 4096), (8, 1040)])
def test_w8a8_small_m_exact_integer(M, K):
    # codes in {-2,-1,-0.5,0,0.5,1,2}: fp32 accumulation is exact; with
    # power-of-two scales the bf16 output equals the rounded exact value
    # (one and two token tiles, K with and without a ragged last chunk)
    vals = {0x40: 2.0, 0x38: 1.0, 0x30: 0.5, 0x00: 0.0, 0xB0: -0.5, 0xB8: -1.0, 0xC0: -2.0}
    codes = np.array(list(vals), np.uint8)
    rng = np.random.default_rng(12 + M + K)
    N = 128
    qa = codes[rng.integers(0, 7, (M, K))]
    qw = codes[rng.integers(0, 7, (N, K))]
    sw = np.array([2.0 ** -(n % 4) for n in range(N)], np.float32)
    y = host(fl.fp8_scaled_mm(dev(qa), dev(qw), scalar(0.5), dev(sw), out_dtype=torch.bfloat16,
                              kernel="stream"))
    exact = oracle.scaled_mm_bruteforce(qa, qw, np.float32(0.5), sw)
    want = torch.from_numpy(exact).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y, want)


@pytest.mark.parametrize("stable", [False, True])
def test_w8a16_chain_with_stable_weights(stable):
    # y1 = x W1^T, then y2 = y1 W2^T on the same stream: with
    # FP8L_WEIGHTS_STABLE the second product starts before the first ends and
    # must still read the finished y1
    M, K, N1, N2 = 16, 4096, 4096, 4096
    x = synthetic.activation(M, K, torch.float16, seed=71)
    w1 = synthetic.weight(N1, K, torch.bfloat16, seed=72)
    w2 = synthetic.weight(N2, N1, torch.bfloat16, seed=73)
    q1, s1 = oracle.quant_per_row(w1)
    q2, s2 = oracle.quant_per_row(w2)
    q1d, s1d, q2d, s2d = dev(q1), dev(s1), dev(q2), dev(s2)
    xd = dev(x)
    for _ in range(3):
        y1 = fl.fp8_w8a16_mm(xd, q1d, s1d, stable_weights=stable)
        y2 = fl.fp8_w8a16_mm(y1, q2d, s2d, stable_weights=stable)
    y1h = host(y1)
    assert_gemm_close(y1h, oracle.w8a16_ref(x, q1, s1))
    y1_f16 = torch.from_numpy(y1h).to(torch.float16)
    assert_gemm_close(host(y2), oracle.w8a16_ref(y1_f16, q2, s2))


@pytest.mark.parametrize("kernel", ["stream", "swapped"])
def test_w8a8_small_m_chain_with_stable_weights(kernel):
    # quantize -> product -> quantize its output -> product, all with the flag
    M, K, N = 8, 4096, 4096
    x = synthetic.activation(M, K, torch.bfloat16, seed=81)
    w1 = synthetic.weight(N, K, torch.bfloat16, seed=82)
    w2 = synthetic.weight(N, N, torch.bfloat16, seed=83)
    q1, s1 = oracle.quant_per_row(w1)
    q2, s2 = oracle.quant_per_row(w2)
    qa, sa = fl.fp8_quant_per_tensor(dev(x))
    y1 = fl.fp8_scaled_mm(qa, dev(q1), sa, dev(s1), out_dtype=torch.bfloat16, stable_weights=True,
                          kernel=kernel)
    qb, sb = fl.fp8_quant_per_tensor(y1)
    y2 = fl.fp8_scaled_mm(qb, dev(q2), sb, dev(s2), out_dtype=torch.bfloat16, stable_weights=True,
                          kernel=kernel)
    qa_o, sa_o = oracle.quant_per_tensor(x)
    assert np.array_equal(host(qa), qa_o)
    assert_gemm_close(host(y1), oracle.scaled_mm_ref(qa_o, q1, sa_o, s1))
    y1_bf16 = torch.from_numpy(host(y1)).to(torch.bfloat16)
    qb_o, sb_o = oracle.quant_per_tensor(y1_bf16)
    assert np.array_equal(host(qb), qb_o) and host(sb)[0] == sb_o
    assert_gemm_close(host(y2), oracle.scaled_mm_ref(qb_o, q2, sb_o, s2))


@pytest.mark.parametrize("kernel", ["stream", "swapped"])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_w8a8_small_m_graph_replay_with_stable_weights(M, kernel):
    # quantize -> product -> quantize -> product in one CUDA graph, the
    # products launched as programmatic dependents: each reads codes and a
    # scale the kernel before it writes.  Every intermediate is zeroed before
    # each replay, so a read that ran ahead of its producer would show.
    K = N = 4096
    x = synthetic.activation(M, K, torch.bfloat16, seed=301 + M)
    q1, s1 = oracle.quant_per_row(synthetic.weight(N, K, torch.bfloat16, seed=302))
    q2, s2 = oracle.quant_per_row(synthetic.weight(N, N, torch.bfloat16, seed=303))
    xd, q1d, s1d, q2d, s2d = dev(x), dev(q1), dev(s1), dev(q2), dev(s2)
    ws = fl.workspace(DEV)
    qa = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    qb = torch.empty((M, N), dtype=torch.uint8, device=DEV)
    sa = torch.empty(1, dtype=torch.float32, device=DEV)
    sb = torch.empty(1, dtype=torch.float32, device=DEV)
    y1 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    y2 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)

    def step():
        fl.fp8_quant_per_tensor(xd, q=qa, scale=sa, ws=ws)
        fl.fp8_scaled_mm(qa, q1d, sa, s1d, out_dtype=torch.bfloat16, y=y1, ws=ws,
                         stable_weights=True, kernel=kernel)
        fl.fp8_quant_per_tensor(y1, q=qb, scale=sb, ws=ws)
        fl.fp8_scaled_mm(qb, q2d, sb, s2d, out_dtype=torch.bfloat16, y=y2, ws=ws,
                         stable_weights=True, kernel=kernel)

    step()
    torch.cuda.synchronize()
    want = y2.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(3):
        for t in (qa, qb, sa, sb, y1, y2):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y2, want)


@pytest.mark.parametrize("M,N", [(1, 4096), (16, 4096), (4, 12288)])
def test_w8a16_graph_replay_with_stable_weights(M, N):
    # two chained products captured in one CUDA graph with the flag: the
    # second is a programmatic dependent of the first (and, for N = 4096, a
    # cluster launch that splits K); the graph must give the eager results
    K = 4096
    x = synthetic.activation(M, K, torch.float16, seed=91 + M)
    w1 = synthetic.weight(N, K, torch.bfloat16, seed=92)
    w2 = synthetic.weight(N, N, torch.bfloat16, seed=93)
    q1, s1 = oracle.quant_per_row(w1)
    q2, s2 = oracle.quant_per_row(w2)
    q1d, s1d, q2d, s2d = dev(q1), dev(s1), dev(q2), dev(s2)
    xd = dev(x)
    y1 = torch.empty((M, N), dtype=torch.float16, device=DEV)
    y2 = torch.empty((M, N), dtype=torch.float16, device=DEV)
    fl.fp8_w8a16_mm(xd, q1d, s1d, y=y1, stable_weights=True)  # set-up outside the capture
    fl.fp8_w8a16_mm(y1, q2d, s2d, y=y2, stable_weights=True)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fl.fp8_w8a16_mm(xd, q1d, s1d, y=y1, stable_weights=True)
        fl.fp8_w8a16_mm(y1, q2d, s2d, y=y2, stable_weights=True)
    want2 = fl.fp8_w8a16_mm(fl.fp8_w8a16_mm(xd, q1d, s1d), q2d, s2d)
    for _ in range(3):
        # zeroed before every replay: a second product that read y1 before
        # the first one finished writing it would see zeros
        y1.zero_()
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y2, want2)
    y1h = host(y1)
    assert_gemm_close(y1h, oracle.w8a16_ref(x, q1, s1))
    assert_gemm_close(host(y2), oracle.w8a16_ref(torch.from_numpy(y1h).to(torch.float16), q2, s2))


@pytest.mark.parametrize("xdtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(16, 9728, 1024), (9, 12288, 512), (16, 22016, 320)])
def test_w8a16_large_n_token_groups(M, N, K, xdtype):
    # 9..16 tokens (two token tiles per CTA) over many channels; K = 320
    # leaves a ragged last 64-k chunk
    y, y_ref = _w8a16_case(M, N, K, xdtype, seed=M + N + K + 5)
    assert_gemm_close(y, y_ref, (M, N, K, xdtype))


@pytest.mark.parametrize("out", ["bf16", "e4m3"])
def test_w8a8_small_m_large_n(out):
    _w8a8_small(16, 10240, 1024, True, out, seed=123, kernel="stream")


def _packed_layout_reference(qw):
    # the packed layout as the header states it: channel n = 16G + 8h + g,
    # k = 64c + 16t + j go to byte (G*C + c)*1024 + h*512 + (4g + t)*16 + j,
    # with zeros for k >= K
    N, K = qw.shape
    C = (K + 63) // 64
    out = np.zeros(N * C * 64, np.uint8)
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    G, h, g = n // 16, (n % 16) // 8, n % 8
    c, t, j = k // 64, (k % 64) // 16, k % 16
    out[(G * C + c) * 1024 + h * 512 + (4 * g + t) * 16 + j] = qw
    return out


@pytest.mark.parametrize("N,K", [(16, 16), (32, 208), (48, 128), (64, 4096), (16, 11008)])
def test_pack_weights_layout(N, K):
    rng = np.random.default_rng(N + K)
    qw = rng.integers(0, 256, (N, K), dtype=np.uint8)
    packed = host(fl.fp8_pack_w8a16_weights(dev(qw)))
    assert packed.dtype == np.uint8 and packed.size == fl.fp8_packed_weight_bytes(N, K)
    assert np.array_equal(packed, _packed_layout_reference(qw))


@pytest.mark.parametrize("xdtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (3, 48, 208), (8, 256, 512), (9, 64, 1024),
                                   (16, 272, 4096), (17, 64, 80), (40, 80, 144),
                                   (16, 4096, 11008)])
def test_w8a16_packed_weights_match_row_major(M, N, K, xdtype):
    # the packed layout only moves the weight bytes: the product is the same
    # bit for bit, and within tolerance of the oracle
    x = synthetic.activation(M, K, xdtype, seed=M + N + K + 17)
    w = synthetic.weight(N, K, torch.bfloat16, seed=M + N + K + 17)
    qw, sw = oracle.quant_per_row(w)
    xd, qwd, swd = dev(x), dev(qw), dev(sw)
    y_rm = fl.fp8_w8a16_mm(xd, qwd, swd)
    y_pk = fl.fp8_w8a16_mm(xd, fl.fp8_pack_w8a16_weights(qwd), swd, packed=True)
    assert torch.equal(y_pk, y_rm)
    assert_gemm_close(host(y_pk), oracle.w8a16_ref(x, qw, sw), (M, N, K, xdtype))


@pytest.mark.parametrize("shape_idx", range(12))
def test_w8a16_decode_workload_packed(shape_idx):
    wl = synthetic.WORKLOADS["decode_w8a16"]
    M, N, K = wl.shapes[shape_idx]
    x = synthetic.activation(M, K, torch.float16, seed=wl.seed(shape_idx))
    w = synthetic.weight(N, K, torch.bfloat16, seed=wl.seed(shape_idx))
    qw, sw = oracle.quant_per_row(w)
    y = fl.fp8_w8a16_mm(dev(x), fl.fp8_pack_w8a16_weights(dev(qw)), dev(sw), packed=True)
    assert_gemm_close(host(y), oracle.w8a16_ref(x, qw, sw), (M, N, K))


def test_w8a16_packed_permutation_weights():
    # every (channel, k) position of the packed layout is paired with the
    # right activation: y[m, n] = sw[n] * x[m, pi(n)] exactly
    K = N = 208
    pi = (np.arange(N) * 37 + 11) % K
    qw = np.zeros((N, K), np.uint8)
    qw[np.arange(N), pi] = 0x38
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    x = synthetic.activation(13, K, torch.float16, seed=19)
    y = host(fl.fp8_w8a16_mm(dev(x), fl.fp8_pack_w8a16_weights(dev(qw)), dev(sw), packed=True))
    want = x.double().numpy()[:, pi] * sw[None, :]
    assert np.array_equal(y, want.astype(np.float16).astype(np.float32))


@pytest.mark.parametrize("M", [1, 16])
def test_w8a16_packed_graph_replay_with_stable_weights(M):
    # two dependent packed products in a CUDA graph, launched as programmatic
    # dependents: the second reads the first one's output
    K = N = 4096
    x = synthetic.activation(M, K, torch.float16, seed=201 + M)
    w1 = synthetic.weight(N, K, torch.bfloat16, seed=202)
    w2 = synthetic.weight(N, K, torch.bfloat16, seed=203)
    q1, s1 = oracle.quant_per_row(w1)
    q2, s2 = oracle.quant_per_row(w2)
    p1, p2 = fl.fp8_pack_w8a16_weights(dev(q1)), fl.fp8_pack_w8a16_weights(dev(q2))
    s1d, s2d, xd = dev(s1), dev(s2), dev(x)
    y1 = torch.empty((M, N), dtype=torch.float16, device=DEV)
    y2 = torch.empty((M, N), dtype=torch.float16, device=DEV)
    want = fl.fp8_w8a16_mm(fl.fp8_w8a16_mm(xd, dev(q1), s1d), dev(q2), s2d)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fl.fp8_w8a16_mm(xd, p1, s1d, y=y1, stable_weights=True, packed=True)
        fl.fp8_w8a16_mm(y1, p2, s2d, y=y2, stable_weights=True, packed=True)
    for _ in range(3):
        y1.zero_()
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y2, want)
