"""The quantizer entry point that allocates nothing.

Some callers cannot allocate device memory: a plug-in that runs inside a
framework owning every device allocation through its own pool, or a serving
loop whose memory footprint is fixed at start-up and that has no workspace to
pass down.  fp8_quant_per_tensor_noalloc keeps its scratch (the per-block
partial maxima and a ticket counter) in an array inside the library image
instead of a caller-provided workspace.

The GPU test calls it through the C ABI on a sequence of tensors, each twice
in a row: a large one first, then smaller ones, so that partial maxima left
over from a larger call are in the array during a smaller one.  The sequence
covers fp32, bf16 and fp16 inputs, element counts that are not a multiple of
16 (the scalar tail), a single element, and an all-zero tensor.  Every call
must give exactly the codes and the scale of the CPU oracle, and of
fp8_quant_per_tensor with a workspace: the quantizer's results are compared
bit for bit everywhere in this test suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import synthetic

_DTYPE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 3}


def _entry(lib):
    f = lib.fp8_quant_per_tensor_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f


def test_rejects_sizes_beyond_the_maximum():
    # checked on the host before any CUDA call
    from fp8_quantized_linear_gb300 import build
    build.build()
    f = _entry(fl.load())
    fake = 0x10000
    assert f(fake, 1, 1 << 30, (1 << 10) + 1, fake, fake, None) == 2  # FP8L_ESHAPE
    assert f(fake, 2, 4, 4, fake, fake, None) == 1                    # FP8L_EINVAL
    assert f(fake + 8, 1, 4, 16, fake, fake, None) == 3               # FP8L_EALIGN


def _inputs():
    yield synthetic.activation(1024, 4096, torch.bfloat16, seed=41, outlier_frac=0.01)
    yield synthetic.activation(3, 4097, torch.float32, seed=43)
    yield synthetic.activation(3, 80, torch.float16, seed=42)
    yield synthetic.activation(7, 13, torch.bfloat16, seed=44)
    yield synthetic.activation(1, 1, torch.float16, seed=45)
    yield torch.zeros((5, 32), dtype=torch.float32)
    yield -synthetic.activation(64, 1000, torch.float32, seed=46) * 1e-3


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls():
    import oracle
    f = _entry(fl.load())
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    for x in _inputs():
        q_o, s_o = oracle.quant_per_tensor(x)
        xd = x.to(dev)
        rows, cols = xd.shape
        q_ws, s_ws = fl.fp8_quant_per_tensor(xd)
        for call in range(2):
            q = torch.full((rows, cols), 0x55, dtype=torch.uint8, device=dev)
            s = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
            st = f(xd.data_ptr(), _DTYPE[xd.dtype], rows, cols, q.data_ptr(), s.data_ptr(),
                   stream.cuda_stream)
            assert st == 0, fl.strerror(st)
            torch.cuda.synchronize(dev)
            what = (tuple(x.shape), x.dtype, call)
            assert np.float32(s.item()).view(np.uint32) == np.float32(s_o).view(np.uint32), what
            assert np.array_equal(q.cpu().numpy(), q_o), what
            assert torch.equal(s, s_ws), what
            assert torch.equal(q, q_ws), what
