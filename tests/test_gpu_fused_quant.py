"""GPU parity of fp8_quant_scaled_mm: the per-tensor activation quantization
fused into the W8A8 product ("Condition to achieve linear speedup?":
quantization fused into another kernel; "RFC: FP8 Quantization Schema in
vLLM": static input scales), in the swapped-operand tcgen05 product or, up
to 16 tokens, the CUDA-core weight stream.  Up to 64 tokens the fused call
must equal, bit for bit, the quantizer followed by the product with the
same kernel choice (same codes, same MMAs, same split of K); its scale and
result must match the CPU oracle: the dynamic scale exactly, the product
within the layer's tolerance."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import DEV, assert_e4m3_close, assert_gemm_close, host, scalar

pytestmark = pytest.mark.gpu


def _status_ok():
    st = fl.fp8l_read_status(fl.workspace(DEV))
    assert st == 0, fl.strerror(st)


def _weights(N, K, per_channel, seed):
    w = synthetic.weight(N, K, torch.bfloat16, seed=seed)
    if per_channel:
        qw, sw = oracle.quant_per_row(w)
    else:
        qw, s = oracle.quant_per_tensor(w)
        sw = np.array([s], np.float32)
    return torch.from_numpy(qw).to(DEV), torch.from_numpy(np.asarray(sw, np.float32)).to(DEV), qw, sw


# dynamic scale: every CTA reads all of x (at most 64 KB); K = 16: one
# partial k-block, 80 and 208: a ragged last one, N = 16 and 48: one partial
# weight block
@pytest.mark.parametrize("kernel", ["auto", "stream", "swapped"])
@pytest.mark.parametrize("xdtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out", ["bf16", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (1, 2320, 14336), (3, 6144, 4096), (16, 512, 2048),
                                   (1, 28672, 4096), (2, 16, 16), (5, 48, 80), (13, 144, 208)])
def test_dynamic_equals_quantizer_then_product(M, N, K, out, xdtype, kernel):
    if kernel == "stream" and M > 16:
        pytest.skip("the weight stream takes up to 16 tokens")
    x = synthetic.activation(M, K, xdtype, seed=M + N + K, outlier_frac=0.01).to(DEV)
    wd, swd, qw, sw = _weights(N, K, out == "e4m3", seed=N)
    os_ = scalar(0.05) if out == "e4m3" else None
    od = torch.uint8 if out == "e4m3" else torch.bfloat16
    # the separate path: quantizer, then the same product kernel
    qa, sa = fl.fp8_quant_per_tensor(x)
    ref_kernel = kernel if kernel != "auto" else (
        "stream" if fl.scaled_mm_kernel(M, N, K) == "stream" else "swapped")
    y_ref = fl.fp8_scaled_mm(qa, wd, sa, swd, out_dtype=od, out_scale=os_, kernel=ref_kernel)
    y, sa_f = fl.fp8_quant_scaled_mm(x, wd, swd, dynamic=True, out_dtype=od, out_scale=os_,
                                     kernel=kernel)
    assert host(sa_f)[0] == host(sa)[0]
    assert torch.equal(y, y_ref)
    # and against the oracle
    qa_o, sa_o = oracle.quant_per_tensor(x.cpu())
    assert np.float32(host(sa_f)[0]) == sa_o
    y_o = oracle.scaled_mm_ref(qa_o, qw, sa_o, sw)
    if out == "e4m3":
        assert_e4m3_close(host(y), y_o, np.float32(0.05))
    else:
        assert_gemm_close(host(y), y_o)
    _status_ok()


# static scale: any M up to 128; values beyond 1024 x scale take the clamp
@pytest.mark.parametrize("stable", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 4096, 8192), (16, 6144, 4096), (64, 10240, 1024), (100, 2320, 640),
                                   (128, 4096, 14336), (4, 4096, 4096), (12, 1024, 2048), (2, 4096, 2048)])
def test_static_equals_quantizer_then_product(M, N, K, stable):
    x = synthetic.activation(M, K, torch.bfloat16, seed=7 * M + K, outlier_frac=0.01).to(DEV)
    wd, swd, qw, sw = _weights(N, K, True, seed=K)
    sa = scalar(float(x.abs().max().item()) / 448.0 * 0.25)  # outliers saturate
    qa = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    fl.fp8_quant_per_tensor(x, q=qa, scale=sa, dynamic=False)
    ref_kernel = "stream" if fl.scaled_mm_kernel(M, N, K) == "stream" else "swapped"
    y_ref = fl.fp8_scaled_mm(qa, wd, sa, swd, out_dtype=torch.bfloat16, kernel=ref_kernel)
    y, _ = fl.fp8_quant_scaled_mm(x, wd, swd, a_scale=sa, dynamic=False, out_dtype=torch.bfloat16,
                                  stable_weights=stable)
    if M <= 64:
        assert torch.equal(y, y_ref)
    else:  # one CTA per SM above 64 tokens: K may be split differently, sums round differently
        assert_gemm_close(host(y), host(y_ref).astype(np.float64))
    qa_o, _ = oracle.quant_per_tensor(x.cpu(), scale=np.float32(host(sa)[0]))
    assert np.array_equal(host(qa).astype(np.uint8), qa_o)
    assert_gemm_close(host(y), oracle.scaled_mm_ref(qa_o, qw, np.float32(host(sa)[0]), sw))
    _status_ok()


_WORKLOAD_CASES = [pytest.param(name, i, id=f"{name}-{M}x{N}x{K}")
                   for name, wl in synthetic.WORKLOADS.items() if wl.kind == "w8a8"
                   for i, (M, N, K) in enumerate(wl.shapes) if M <= 16]


@pytest.mark.parametrize("name,i", _WORKLOAD_CASES)
def test_workload_shapes_where_fused_is_preferred(name, i):
    # every product the benchmark runs as one fused call: its workload's
    # activations, scale mode, weight scales and output type
    wl = synthetic.WORKLOADS[name]
    M, N, K = wl.shapes[i]
    dynamic = wl.act_scale == "dynamic"
    if not fl.quant_scaled_mm_preferred(M, N, K, dynamic):
        pytest.skip("quantizer + product is the faster path for this shape")
    x = synthetic.activation(M, K, wl.x_dtype, seed=wl.seed(i), outlier_frac=wl.outlier_frac).to(DEV)
    wd, swd, qw, sw = _weights(N, K, wl.w_scale == "channel", seed=wl.seed(i))
    if dynamic:
        qa_o, sa_o = oracle.quant_per_tensor(x.cpu())
        sa = torch.empty(1, dtype=torch.float32, device=DEV)
    else:
        sa_o = np.float32(float(x.abs().max().item()) / 448.0 * 0.75)  # the outliers saturate
        qa_o, _ = oracle.quant_per_tensor(x.cpu(), scale=sa_o)
        sa = scalar(sa_o)
    y_o = oracle.scaled_mm_ref(qa_o, qw, sa_o, sw)
    e4m3 = wl.out_dtype == "e4m3"
    od = {"bf16": torch.bfloat16, "fp16": torch.float16, "e4m3": torch.uint8}[wl.out_dtype]
    os_v = np.float32(np.abs(y_o).max() / 448.0) if e4m3 else None
    os_ = scalar(os_v) if e4m3 else None
    y, sa_f = fl.fp8_quant_scaled_mm(x, wd, swd, a_scale=sa, dynamic=dynamic, out_dtype=od,
                                     out_scale=os_, stable_weights=True)
    assert np.float32(host(sa_f)[0]) == np.float32(sa_o)
    qa = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    sa2 = torch.empty(1, dtype=torch.float32, device=DEV) if dynamic else sa
    fl.fp8_quant_per_tensor(x, q=qa, scale=sa2, dynamic=dynamic)
    assert np.array_equal(host(qa).astype(np.uint8), qa_o)
    ref_kernel = "stream" if fl.scaled_mm_kernel(M, N, K) == "stream" else "swapped"
    y_sep = fl.fp8_scaled_mm(qa, wd, sa2, swd, out_dtype=od, out_scale=os_, kernel=ref_kernel)
    assert torch.equal(y, y_sep)
    if e4m3:
        assert_e4m3_close(host(y), y_o, os_v)
    else:
        assert_gemm_close(host(y), y_o)
    _status_ok()


@pytest.mark.parametrize("kernel", ["stream", "swapped"])
def test_graph_chain(kernel):
    # x -> y1 (dynamic) -> y2 = fused(y1) (dynamic) in one CUDA graph, both
    # programmatic dependents; outputs and scales zeroed before each replay
    M, K, N = 1, 4096, 4096
    x = synthetic.activation(M, K, torch.bfloat16, seed=91).to(DEV)
    w1, s1, q1, sw1 = _weights(N, K, True, seed=92)
    w2, s2, q2, sw2 = _weights(N, N, True, seed=93)
    y1 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    y2 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    a1 = torch.empty(1, dtype=torch.float32, device=DEV)
    a2 = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = fl.workspace(DEV)

    def step():
        fl.fp8_quant_scaled_mm(x, w1, s1, a_scale=a1, y=y1, ws=ws, stable_weights=True, kernel=kernel)
        fl.fp8_quant_scaled_mm(y1, w2, s2, a_scale=a2, y=y2, ws=ws, stable_weights=True, kernel=kernel)

    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    want1, want2 = y1.clone(), y2.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(3):
        for t in (y1, y2, a1, a2):
            t.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1, want1) and torch.equal(y2, want2)
    qa_o, sa_o = oracle.quant_per_tensor(x.cpu())
    assert_gemm_close(host(y1), oracle.scaled_mm_ref(qa_o, q1, sa_o, sw1))
    _status_ok()


def test_bounds():
    w = torch.zeros((64, 64), dtype=torch.uint8, device=DEV)
    s = torch.ones(1, dtype=torch.float32, device=DEV)
    with pytest.raises(RuntimeError):  # more than 128 tokens
        fl.fp8_quant_scaled_mm(torch.zeros((129, 64), dtype=torch.bfloat16, device=DEV), w, s)
    with pytest.raises(RuntimeError):  # the weight stream takes up to 16 tokens
        fl.fp8_quant_scaled_mm(torch.zeros((17, 64), dtype=torch.bfloat16, device=DEV), w, s,
                               kernel="stream")
    with pytest.raises(RuntimeError):  # dynamic x larger than 64 KB
        fl.fp8_quant_scaled_mm(torch.zeros((64, 1024), dtype=torch.bfloat16, device=DEV),
                               torch.zeros((64, 1024), dtype=torch.uint8, device=DEV), s)
    y, _ = fl.fp8_quant_scaled_mm(torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV), w, s)
    assert y.shape == (0, 64)
