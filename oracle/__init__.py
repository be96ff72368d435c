"""CPU oracle for the FP8 E4M3 quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's ``smoke()`` check
and the benchmark's CPU-baseline leg may import this package.  The GPU library
does not import it, and it imports nothing from the GPU library: the two share
no code.  Inputs come from the separate ``synthetic`` module.

The arithmetic lives in ``fp8_oracle.c`` (plain loops, double accumulation,
built with ``-O2 -fno-fast-math -ffp-contract=off``).  This module adds
marshalling, exact widening of 16-bit inputs to fp32, and one library
primitive: a float64 matrix product of the decoded operands (numpy) for shapes
too large for the brute-force loops.  The tests pin that product against the
brute-force C loops on small shapes.

What each function follows (page title, then the part of the page):
  * E4M3 decode/encode: "RFC: FP8 Quantization Schema in vLLM", Scope (OCP
    FP8_E4M3); "[Kernel][FP8] Initial support with dynamic per-tensor
    scaling", the ``torch.float8_e4m3fn`` cast of the microbenchmark list.
  * per-tensor quantization: "[Kernel][FP8] Initial support ...", Algorithm.
  * per-channel weight scale: "Marlin fp8", kernel argument checks
    (``b_scales`` of shape [1, N]).
  * static input / output scale: "RFC: FP8 Quantization Schema in vLLM",
    Interface Content, and the ``output_scale`` discussion after it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfp8oracle.so")

_lock = threading.Lock()
_lib = None

E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain IEEE arithmetic, no contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.fp8o_e4m3_decode.argtypes = [ctypes.c_uint]
        lib.fp8o_e4m3_decode.restype = ctypes.c_double
        lib.fp8o_e4m3_decode_table.argtypes = [P]
        lib.fp8o_e4m3_encode.argtypes = [ctypes.c_double]
        lib.fp8o_e4m3_encode.restype = ctypes.c_uint
        lib.fp8o_e4m3_encode_f64_array.argtypes = [P, I64, P]
        lib.fp8o_e4m3_encode_f32_array.argtypes = [P, I64, P]
        lib.fp8o_amax.argtypes = [P, I64]
        lib.fp8o_amax.restype = ctypes.c_float
        lib.fp8o_scale_from_amax.argtypes = [ctypes.c_float]
        lib.fp8o_scale_from_amax.restype = ctypes.c_float
        lib.fp8o_quant_with_scale.argtypes = [P, I64, ctypes.c_float, P]
        lib.fp8o_quant_per_tensor.argtypes = [P, I64, P, P]
        lib.fp8o_quant_per_row.argtypes = [P, I64, I64, P, P]
        lib.fp8o_scaled_mm_f64.argtypes = [P, P, I64, I64, I64, ctypes.c_float,
                                           P, ctypes.c_int, P]
        lib.fp8o_w8a16_mm_f64.argtypes = [P, P, P, I64, I64, I64, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# --------------------------------------------------------------------------
# E4M3 format

def decode_table() -> np.ndarray:
    """float64 value of every code 0..255 (NaN at 0x7F and 0xFF)."""
    out = np.empty(256, dtype=np.float64)
    _load().fp8o_e4m3_decode_table(_ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    return decode_table()[codes]


def e4m3_encode(values) -> np.ndarray:
    """Saturating round-to-nearest-even encode of each value (float32 values
    are encoded as they are; float64 values are encoded without first
    rounding them to float32)."""
    v = np.asarray(values)
    lib = _load()
    if v.dtype == np.float32:
        v = np.ascontiguousarray(v)
        out = np.empty(v.shape, dtype=np.uint8)
        lib.fp8o_e4m3_encode_f32_array(_ptr(v), v.size, _ptr(out))
    else:
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint8)
        lib.fp8o_e4m3_encode_f64_array(_ptr(v), v.size, _ptr(out))
    return out


# --------------------------------------------------------------------------
# inputs

def widen(x) -> np.ndarray:
    """Exact float32 copy of a bf16 / fp16 / fp32 tensor or array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype not in (torch.bfloat16, torch.float16, torch.float32):
                raise TypeError(f"unsupported dtype {x.dtype}")
            return np.ascontiguousarray(x.float().numpy())
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype not in (np.float16, np.float32):
        raise TypeError(f"unsupported dtype {x.dtype}")
    return np.ascontiguousarray(x.astype(np.float32))


# --------------------------------------------------------------------------
# quantization

def amax(x) -> np.float32:
    xf = widen(x)
    return np.float32(_load().fp8o_amax(_ptr(xf), xf.size))


def scale_from_amax(a) -> np.float32:
    return np.float32(_load().fp8o_scale_from_amax(float(np.float32(a))))


def quant_per_tensor(x, scale=None):
    """Per-tensor quantization.  With ``scale=None`` the scale is dynamic
    (amax / 448); otherwise the given static scale is used.  Returns
    ``(codes uint8 with x's shape, scale float32)``."""
    xf = widen(x)
    q = np.empty(xf.shape, dtype=np.uint8)
    lib = _load()
    if scale is None:
        s = np.zeros(1, dtype=np.float32)
        lib.fp8o_quant_per_tensor(_ptr(xf), xf.size, _ptr(q), _ptr(s))
        return q, np.float32(s[0])
    s = np.float32(scale)
    lib.fp8o_quant_with_scale(_ptr(xf), xf.size, float(s), _ptr(q))
    return q, s


def quant_per_row(w):
    """One dynamic scale per row of a 2-D tensor.  Returns (codes, scales[rows])."""
    wf = widen(w)
    assert wf.ndim == 2
    rows, cols = wf.shape
    q = np.empty(wf.shape, dtype=np.uint8)
    s = np.empty(rows, dtype=np.float32)
    _load().fp8o_quant_per_row(_ptr(wf), rows, cols, _ptr(q), _ptr(s))
    return q, s


# --------------------------------------------------------------------------
# matrix products

def _scales(sw, N):
    sw = np.ascontiguousarray(np.asarray(sw, dtype=np.float32).reshape(-1))
    if sw.size not in (1, N):
        raise ValueError("weight scale must have 1 or N entries")
    return sw


def scaled_mm_bruteforce(qa, qw, sa, sw) -> np.ndarray:
    """y = (sa * sw[n]) * sum_k dec(qa[m,k]) dec(qw[n,k]) by triple loop (C)."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    M, K = qa.shape
    N, K2 = qw.shape
    assert K == K2
    sw = _scales(sw, N)
    y = np.empty((M, N), dtype=np.float64)
    _load().fp8o_scaled_mm_f64(_ptr(qa), _ptr(qw), M, N, K, float(np.float32(sa)),
                               _ptr(sw), int(sw.size == N and N != 1), _ptr(y))
    return y


def scaled_mm_ref(qa, qw, sa, sw) -> np.ndarray:
    """Same result as ``scaled_mm_bruteforce`` through a float64 matrix product
    of the decoded operands (library primitive; pinned against the loops)."""
    table = decode_table()
    A = table[np.asarray(qa, dtype=np.uint8)]
    W = table[np.asarray(qw, dtype=np.uint8)]
    N = W.shape[0]
    sw = _scales(sw, N).astype(np.float64)
    acc = A @ W.T
    return acc * (np.float64(np.float32(sa)) * sw.reshape(1, -1))


def w8a16_bruteforce(x, qw, sw) -> np.ndarray:
    """y = sw[n] * sum_k x[m,k] dec(qw[n,k]) by triple loop (C)."""
    xf = widen(x)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    M, K = xf.shape
    N, K2 = qw.shape
    assert K == K2
    sw = np.ascontiguousarray(np.asarray(sw, dtype=np.float32).reshape(-1))
    assert sw.size == N
    y = np.empty((M, N), dtype=np.float64)
    _load().fp8o_w8a16_mm_f64(_ptr(xf), _ptr(qw), _ptr(sw), M, N, K, _ptr(y))
    return y


def w8a16_ref(x, qw, sw) -> np.ndarray:
    """``w8a16_bruteforce`` through a float64 matrix product (library primitive)."""
    X = widen(x).astype(np.float64)
    W = decode_table()[np.asarray(qw, dtype=np.uint8)]
    sw = np.asarray(sw, dtype=np.float32).reshape(-1).astype(np.float64)
    assert sw.size == W.shape[0]
    return (X @ W.T) * sw.reshape(1, -1)


def e4m3_output_ref(y_ref, out_scale) -> np.ndarray:
    """Reference E4M3 output codes: E4M3(y_ref / output_scale) with the
    quotient kept in float64 (no intermediate float32 rounding)."""
    y = np.asarray(y_ref, dtype=np.float64)
    return e4m3_encode(y / np.float64(np.float32(out_scale)))
