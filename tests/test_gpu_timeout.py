"""Failure detection on the GPU without a fault: every device-side wait of the
tcgen05 product and of the dynamic quantizer is bounded.  The testing hook
fp8l_debug_waits shortens the limit (about half a millisecond here) and makes
one wait target a barrier that nothing completes; the call must record
FP8L_ETIMEOUT, return without hanging, leave the context usable, and
fp8l_read_status must reset the workspace so that the next ordinary call is
exact again (compared with the CPU oracle)."""
import numpy as np
import pytest
import torch

import fp8_quantized_linear_gb300 as fl
import oracle
import synthetic
from gpu_util import DEV, assert_gemm_close, host, scaled_mm_ref_rows

pytestmark = pytest.mark.gpu

SHORT = 1 << 20  # cycles


@pytest.fixture(autouse=True)
def restore_defaults():
    yield
    fl.fp8l_debug_waits(0, 0)


def _operands(M, N, K, seed):
    x = synthetic.activation(M, K, torch.bfloat16, seed=seed)
    w = synthetic.weight(N, K, torch.bfloat16, seed=seed)
    qa, sa = oracle.quant_per_tensor(x)
    qw, sw = oracle.quant_per_tensor(w)
    return qa, sa, qw, sw


# persistent tiles; cluster split-K; swapped operands with and without a
# cluster splitting K
@pytest.mark.parametrize("M,kernel", [(256, "auto"), (64, "auto"), (64, "swapped"), (8, "swapped")])
def test_product_wait_times_out_then_recovers(M, kernel):
    N, K = 512, 1024
    qa, sa, qw, sw = _operands(M, N, K, seed=900 + M)
    ws = fl.workspace(DEV)
    assert fl.fp8l_read_status(ws) == fl._binding.OK
    a, w = torch.from_numpy(qa).to(DEV), torch.from_numpy(qw).to(DEV)
    sa_d = torch.tensor([sa], dtype=torch.float32, device=DEV)
    sw_d = torch.tensor([sw], dtype=torch.float32, device=DEV)
    fl.fp8l_debug_waits(SHORT, fl._binding.STALL_MMA)
    fl.fp8_scaled_mm(a, w, sa_d, sw_d, out_dtype=torch.bfloat16, ws=ws, kernel=kernel)
    torch.cuda.synchronize()
    assert fl.fp8l_read_status(ws) == fl._binding.ETIMEOUT
    # the workspace was reset with the status: the next ordinary call is exact
    fl.fp8l_debug_waits(0, 0)
    y = fl.fp8_scaled_mm(a, w, sa_d, sw_d, out_dtype=torch.bfloat16, ws=ws, kernel=kernel)
    assert fl.fp8l_read_status(ws) == fl._binding.OK
    y_ref = scaled_mm_ref_rows(qa, qw, sa, [sw])
    assert_gemm_close(host(y), y_ref, "after a time-out")


def test_w8a16_tensor_core_wait_times_out_then_recovers():
    # fp8_w8a16_mm takes no workspace: its tensor-core kernel records the
    # time-out in the library's status word, which fp8l_read_status reports
    # and clears with the workspace's
    M, N, K = 16, 512, 1024
    x = synthetic.activation(M, K, torch.float16, seed=913)
    qw, sw = oracle.quant_per_row(synthetic.weight(N, K, torch.bfloat16, seed=914))
    xd, wd, sd = x.to(DEV), torch.from_numpy(qw).to(DEV), torch.from_numpy(sw).to(DEV)
    ws = fl.workspace(DEV)
    assert fl.fp8l_read_status(ws) == fl._binding.OK
    fl.fp8l_debug_waits(SHORT, fl._binding.STALL_MMA)
    fl.fp8_w8a16_mm(xd, wd, sd, kernel="swapped")
    torch.cuda.synchronize()
    assert fl.fp8l_read_status(ws) == fl._binding.ETIMEOUT
    assert fl.fp8l_read_status(ws) == fl._binding.OK  # reported once, then cleared
    fl.fp8l_debug_waits(0, 0)
    y = fl.fp8_w8a16_mm(xd, wd, sd, kernel="swapped")
    assert fl.fp8l_read_status(ws) == fl._binding.OK
    assert_gemm_close(host(y), oracle.w8a16_ref(x, qw, sw), "after a time-out")


def test_quantizer_grid_barrier_times_out_then_recovers():
    x = synthetic.activation(1024, 4096, torch.bfloat16, seed=907, outlier_frac=0.01)
    q_o, s_o = oracle.quant_per_tensor(x)
    xd = x.to(DEV)
    ws = fl.workspace(DEV)
    assert fl.fp8l_read_status(ws) == fl._binding.OK
    fl.fp8l_debug_waits(SHORT, fl._binding.STALL_GRID)
    fl.fp8_quant_per_tensor(xd, ws=ws)
    torch.cuda.synchronize()
    assert fl.fp8l_read_status(ws) == fl._binding.ETIMEOUT
    fl.fp8l_debug_waits(0, 0)
    for _ in range(3):  # both barrier-word pairs are used again
        q, s = fl.fp8_quant_per_tensor(xd, ws=ws)
        assert fl.fp8l_read_status(ws) == fl._binding.OK
        assert np.float32(s.item()) == s_o
        assert np.array_equal(q.cpu().numpy(), q_o)


def test_short_limit_alone_does_not_time_out():
    # a limit of ~0.5 ms is far above any healthy wait of these small calls
    qa, sa, qw, sw = _operands(256, 512, 1024, seed=911)
    ws = fl.workspace(DEV)
    fl.fp8l_debug_waits(SHORT, 0)
    a, w = torch.from_numpy(qa).to(DEV), torch.from_numpy(qw).to(DEV)
    sa_d = torch.tensor([sa], dtype=torch.float32, device=DEV)
    sw_d = torch.tensor([sw], dtype=torch.float32, device=DEV)
    y = fl.fp8_scaled_mm(a, w, sa_d, sw_d, out_dtype=torch.bfloat16, ws=ws)
    x = synthetic.activation(256, 1024, torch.bfloat16, seed=912)
    q, s = fl.fp8_quant_per_tensor(x.to(DEV), ws=ws)
    assert fl.fp8l_read_status(ws) == fl._binding.OK
    assert_gemm_close(host(y), scaled_mm_ref_rows(qa, qw, sa, [sw]))
    q_o, s_o = oracle.quant_per_tensor(x)
    assert np.array_equal(q.cpu().numpy(), q_o) and np.float32(s.item()) == s_o
