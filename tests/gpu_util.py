"""Helpers shared by the GPU parity tests (CUDA path vs CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

DEV = torch.device("cuda:0")


def dev(a) -> torch.Tensor:
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a))
    elif not isinstance(a, torch.Tensor):
        a = torch.tensor(a)
    return a.to(DEV)


def scalar(v) -> torch.Tensor:
    return torch.tensor([float(np.float32(v))], dtype=torch.float32, device=DEV)


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.cpu().numpy()


def assert_status_ok():
    import fp8_quantized_linear_gb300 as fl
    st = fl.fp8l_read_status(fl.workspace(DEV))
    assert st == 0, fl.strerror(st)


def scaled_mm_ref_rows(qa_rows, qw, sa, sw, n_block=4096):
    """float64 reference for some rows of A, computed in column blocks of W
    to bound host memory."""
    table = oracle.decode_table()
    A = table[qa_rows]
    N = qw.shape[0]
    sw = np.asarray(sw, np.float32).reshape(-1)
    out = np.empty((A.shape[0], N), np.float64)
    for n0 in range(0, N, n_block):
        n1 = min(N, n0 + n_block)
        out[:, n0:n1] = oracle.scaled_mm_ref(qa_rows, qw[n0:n1], sa,
                                             sw if sw.size == 1 else sw[n0:n1])
    return out


def assert_gemm_close(y, y_ref, what=""):
    res = oracle.gemm_close(y, y_ref)
    assert res["ok"], (what, res)
    return res


def assert_e4m3_close(codes, y_ref, out_scale, what=""):
    res = oracle.e4m3_output_close(codes, y_ref, out_scale)
    assert res["ok"], (what, res)
    return res


def sample_rows(M: int, count: int, seed: int) -> np.ndarray:
    """Seeded row sample that always includes the first and the last row."""
    if M <= count:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    rows = rng.choice(M, size=count - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], rows]))
