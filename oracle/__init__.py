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
  * per-token activation scales (one per row of the activation codes): the
    RFC's Scope, which leaves scales finer than per-tensor for later; read
    as one scale per activation row.
  * grouped products for mixture-of-experts layers: "RFC: FP8 Quantization
    Schema in vLLM", the gate_proj question (FP8 products need shapes
    divisible by 16; the experts' products are FP8).
  * RMS normalization before the quantizer: "Condition to achieve linear
    speedup?", where the activation quantization is fused into an
    element-wise kernel such as RMSNorm; the pages do not define RMSNorm,
    so the plain (Llama) definition is used, its output stored in the
    activation's 16-bit format, then quantized as above.
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
        lib.fp8o_scaled_mm_rows_f64.argtypes = [P, P, I64, I64, I64, P, P, ctypes.c_int, P]
        lib.fp8o_w8a16_mm_f64.argtypes = [P, P, P, I64, I64, I64, P]
        lib.fp8o_rmsnorm_f64.argtypes = [P, P, I64, I64, ctypes.c_double, P]
        lib.fp8o_grouped_mm_f64.argtypes = [P, P, P, I64, I64, I64, I64, P, ctypes.c_int, P,
                                            ctypes.c_int, P]
        lib.fp8o_round_binary.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int]
        lib.fp8o_round_binary.restype = ctypes.c_double
        lib.fp8o_round_binary_array.argtypes = [P, I64, ctypes.c_int, ctypes.c_int, P]
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


def _act_scales(sa, M):
    sa = np.ascontiguousarray(np.asarray(sa, dtype=np.float32).reshape(-1))
    if sa.size not in (1, M):
        raise ValueError("activation scale must have 1 or M entries")
    return sa


def scaled_mm_bruteforce(qa, qw, sa, sw) -> np.ndarray:
    """y = (sa * sw[n]) * sum_k dec(qa[m,k]) dec(qw[n,k]) by triple loop (C).
    sa is one per-tensor scale, or M per-row (per-token) scales sa[m]."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    M, K = qa.shape
    N, K2 = qw.shape
    assert K == K2
    sw = _scales(sw, N)
    sa = _act_scales(sa, M)
    y = np.empty((M, N), dtype=np.float64)
    per_channel = int(sw.size == N and N != 1)
    if sa.size == 1:
        _load().fp8o_scaled_mm_f64(_ptr(qa), _ptr(qw), M, N, K, float(sa[0]), _ptr(sw),
                                   per_channel, _ptr(y))
    else:
        _load().fp8o_scaled_mm_rows_f64(_ptr(qa), _ptr(qw), M, N, K, _ptr(sa), _ptr(sw),
                                        per_channel, _ptr(y))
    return y


def scaled_mm_ref(qa, qw, sa, sw) -> np.ndarray:
    """Same result as ``scaled_mm_bruteforce`` through a float64 matrix product
    of the decoded operands (library primitive; pinned against the loops)."""
    table = decode_table()
    A = table[np.asarray(qa, dtype=np.uint8)]
    W = table[np.asarray(qw, dtype=np.uint8)]
    N = W.shape[0]
    sw = _scales(sw, N).astype(np.float64)
    sa = _act_scales(sa, A.shape[0]).astype(np.float64)
    acc = A @ W.T
    return acc * (sa.reshape(-1, 1) * sw.reshape(1, -1))


def grouped_mm_bruteforce(qa, qw, offsets, sa, sw) -> np.ndarray:
    """Grouped product by loops (C): rows offsets[e] .. offsets[e+1]-1 of qa
    use expert e's weights qw[e] [N, K] and scales sw[e] (one, or N).
    Rows outside every group are left 0."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    offs = np.ascontiguousarray(offsets, dtype=np.int32)
    M, K = qa.shape
    E, N, K2 = qw.shape
    assert K == K2 and offs.size == E + 1
    sw = np.ascontiguousarray(np.asarray(sw, np.float32).reshape(E, -1))
    assert sw.shape[1] in (1, N)
    sa = _act_scales(sa, M)
    y = np.zeros((M, N), dtype=np.float64)
    _load().fp8o_grouped_mm_f64(_ptr(qa), _ptr(qw), _ptr(offs), E, M, N, K, _ptr(sa),
                                int(sa.size == M and M != 1), _ptr(sw),
                                int(sw.shape[1] == N and N != 1), _ptr(y))
    return y


def grouped_mm_ref(qa, qw, offsets, sa, sw) -> np.ndarray:
    """``grouped_mm_bruteforce`` through one float64 matrix product per
    expert (library primitive)."""
    qa = np.asarray(qa, dtype=np.uint8)
    E, N, _ = np.asarray(qw).shape
    M = qa.shape[0]
    sw = np.asarray(sw, np.float32).reshape(E, -1)
    sa = _act_scales(sa, M).astype(np.float64)
    y = np.zeros((M, N), np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), min(int(offsets[e + 1]), M)
        if hi <= lo:
            continue
        rows_sa = sa[lo:hi] if sa.size == M and M != 1 else sa[:1]
        y[lo:hi] = scaled_mm_ref(qa[lo:hi], qw[e], rows_sa if rows_sa.size > 1 else rows_sa[0],
                                 sw[e] if sw.shape[1] == N else sw[e, :1])
    return y


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


# --------------------------------------------------------------------------
# RMS normalization feeding the quantizer

# (significand bits with the implicit one, minimum normal exponent)
FORMATS = {"bf16": (8, -126), "fp16": (11, -14)}


def _fmt(dtype) -> str:
    name = str(dtype).replace("torch.", "")
    return {"bfloat16": "bf16", "float16": "fp16", "bf16": "bf16", "fp16": "fp16"}[name]


def rmsnorm_ref(x, gamma, eps) -> np.ndarray:
    """h = x * gamma / sqrt(mean_k x^2 + eps) per row, in float64 (C loops)."""
    xf = widen(x)
    gf = widen(gamma).reshape(-1)
    assert xf.ndim == 2 and gf.size == xf.shape[1]
    h = np.empty(xf.shape, np.float64)
    _load().fp8o_rmsnorm_f64(_ptr(xf), _ptr(np.ascontiguousarray(gf)), xf.shape[0], xf.shape[1],
                             float(eps), _ptr(h))
    return h


def round_to(v, dtype) -> np.ndarray:
    """Round float64 values to the nearest bf16 / fp16 value (ties to even,
    gradual underflow), returned as float64."""
    p, emin = FORMATS[_fmt(dtype)]
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.float64)
    _load().fp8o_round_binary_array(_ptr(v), v.size, p, emin, _ptr(out))
    return out


def rmsnorm_quant(x, gamma, eps, mode="tensor", scale=None):
    """The layer's normalization followed by quantization, as the unfused
    layer computes it: h = RMSNorm(x) stored in x's 16-bit format, then
    per-tensor (dynamic or static) or per-row quantization of h.  Returns
    (codes, scale(s), h as float64 of the 16-bit values)."""
    import torch
    dt = x.dtype if isinstance(x, torch.Tensor) else x
    h = round_to(rmsnorm_ref(x, gamma, eps), dt)
    h32 = h.astype(np.float32)  # exact: every 16-bit value is a float32
    if mode == "row":
        q, s = quant_per_row(h32)
    elif mode == "tensor":
        q, s = quant_per_tensor(h32, scale)
    else:
        raise ValueError(mode)
    return q, s, h


# --------------------------------------------------------------------------
# parity criteria (used by the tests, the smoke check and the benchmark)

GEMM_ELEMENT_TOL = 1e-2   # |y - y_ref| <= 1e-2 (|y_ref| + rms(y_ref)) per element
GEMM_FRO_TOL = 5e-3       # ||y - y_ref||_F <= 5e-3 ||y_ref||_F
E4M3_FRO_TOL = 2.0 ** -4  # E4M3 output: half the relative code spacing
E4M3_MIDPOINT_WINDOW = 1e-3


def gemm_close(y, y_ref) -> dict:
    """Tolerance of a 16-bit GEMM output against the float64 reference of
    the same FP8 operands: elementwise ``|y - y_ref| <= 1e-2 (|y_ref| +
    rms(y_ref))`` and relative Frobenius error ``<= 5e-3``."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape
    if y.size == 0:
        return {"ok": True, "max_ratio": 0.0, "rel_fro": 0.0}
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    err = np.abs(y - y_ref)
    bound = GEMM_ELEMENT_TOL * (np.abs(y_ref) + rms)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    max_ratio = float(np.max(ratio))
    nref = float(np.linalg.norm(y_ref))
    rel_fro = float(np.linalg.norm(y - y_ref) / nref) if nref > 0 else float(np.linalg.norm(y))
    ok = bool(np.all(np.isfinite(y))) and max_ratio <= 1.0 and rel_fro <= GEMM_FRO_TOL
    return {"ok": ok, "max_ratio": max_ratio, "rel_fro": rel_fro}


NORM_MIDPOINT_WINDOW = 2.0 ** -16  # relative; see rounded_close


def rounded_close(h, h_ref, dtype, window=NORM_MIDPOINT_WINDOW) -> dict:
    """Tolerance of a 16-bit result h computed in float32 against the
    float64 reference h_ref of the same operation: h must be the rounding
    of h_ref to the format (ties to even), except where h_ref lies within
    ``window * |h_ref|`` of a rounding midpoint, where either neighbour is
    accepted.  The window covers the float32 evaluation's relative error
    (below 2^-17 for a sum of at most 2^16 squares, a square root, a
    reciprocal and two products)."""
    p, emin = FORMATS[_fmt(dtype)]
    h = np.asarray(h, np.float64)
    h_ref = np.asarray(h_ref, np.float64)
    assert h.shape == h_ref.shape
    want = round_to(h_ref, dtype)
    lo = round_to(h_ref * (1 - window), dtype)
    hi = round_to(h_ref * (1 + window), dtype)
    exact = h == want
    either = (h == lo) | (h == hi)
    ok_each = exact | either
    bad = int(np.count_nonzero(~ok_each | ~np.isfinite(h)))
    return {"ok": bad == 0, "bad": bad, "differing": int(np.count_nonzero(~exact))}


def _signed_ordinal(codes):
    c = np.asarray(codes, dtype=np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def _nearest_midpoint_distance(t):
    pos = decode_table()[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    a = np.minimum(np.abs(t), 448.0)
    i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    return np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))


def e4m3_output_close(codes, y_ref, out_scale) -> dict:
    """Tolerance of an E4M3 GEMM output (codes) against y_ref.

    Reading (the stated GEMM tolerance is finer than E4M3 can resolve):
    c_ref = E4M3(y_ref / out_scale) in float64; every code is within one
    step of c_ref on the signed code ordinal (0x00 and 0x80 equal);
    codes equal c_ref wherever t = y_ref / out_scale lies farther than
    1e-3 (|t| + rms(t)) from a rounding midpoint; and
    ||dec(code) - clip(t)||_F <= 2^-4 ||clip(t)||_F with clip to +-448
    (the saturated reference)."""
    codes = np.asarray(codes, dtype=np.uint8)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    os_ = np.float64(np.float32(out_scale))
    t = y_ref / os_
    c_ref = e4m3_encode(t)
    step = np.abs(_signed_ordinal(codes) - _signed_ordinal(c_ref))
    rms = float(np.sqrt(np.mean(t ** 2))) if t.size else 0.0
    far = _nearest_midpoint_distance(t) > E4M3_MIDPOINT_WINDOW * (np.abs(t) + rms)
    exact_bad = int(np.count_nonzero(far & (_signed_ordinal(codes) != _signed_ordinal(c_ref))))
    tc = np.clip(t, -448.0, 448.0)
    dec = decode_table()[codes]
    nref = float(np.linalg.norm(tc))
    rel_fro = float(np.linalg.norm(dec - tc) / nref) if nref > 0 else float(np.linalg.norm(dec))
    max_step = int(step.max()) if step.size else 0
    ok = max_step <= 1 and exact_bad == 0 and rel_fro <= E4M3_FRO_TOL and not np.any(np.isnan(dec))
    return {"ok": ok, "max_step": max_step, "exact_mismatch": exact_bad, "rel_fro": rel_fro,
            "differing": int(np.count_nonzero(step))}
