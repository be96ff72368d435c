"""The quantizer entry point that allocates nothing.

Some callers cannot allocate device memory: a plug-in that runs inside a
framework owning every device allocation through its own pool, or a serving
loop whose memory footprint is fixed at start-up and that has no workspace to
pass down.  fp8_quant_per_tensor_noalloc keeps its scratch (the per-block
partial maxima) in an array inside the library image instead of a
caller-provided workspace.

The GPU test calls it through the C ABI twice in a row (a large tensor, then a
small one, so entries left over from the first call are in the array during
the second) and checks that each call returns exactly the codes and the scale
of fp8_quant_per_tensor with a workspace: the quantizer's results are
compared bit for bit everywhere in this test suite.
"""
import ctypes

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


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    f = _entry(fl.load())
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    inputs = [synthetic.activation(1024, 4096, torch.bfloat16, seed=41, outlier_frac=0.01),
              synthetic.activation(3, 80, torch.float16, seed=42)]
    for x in inputs:
        xd = x.to(dev)
        rows, cols = xd.shape
        q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        s = torch.empty(1, dtype=torch.float32, device=dev)
        st = f(xd.data_ptr(), _DTYPE[xd.dtype], rows, cols, q.data_ptr(), s.data_ptr(),
               stream.cuda_stream)
        assert st == 0, fl.strerror(st)
        q_ref, s_ref = fl.fp8_quant_per_tensor(xd)
        torch.cuda.synchronize(dev)
        assert torch.equal(s, s_ref), (s.item(), s_ref.item())
        assert torch.equal(q, q_ref)
