"""ctypes binding of libfp8linear.so: argument marshalling only.

Every function has the name of the C entry point it calls.  Tensors are torch
CUDA tensors (torch supplies device memory and the current stream); E4M3
tensors are uint8 code tensors (a torch.float8_e4m3fn tensor is accepted and
viewed as uint8).  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8linear.so")

ABI_VERSION = 7  # the library version this binding is written for
F16, BF16, E4M3, F32 = 0, 1, 2, 3
WEIGHTS_STABLE = 1
WEIGHTS_PACKED = 2
A_PER_TOKEN = 4
SINGLE_SM_TILES = 8
KERNELS = {"auto": 0, "stream": 16, "swapped": 32, "tiled": 48}  # FP8L_KERNEL_*
FUSED_DYNAMIC_MAX_BYTES = 65536  # FP8L_FUSED_DYNAMIC_MAX_BYTES
OK, EINVAL, ESHAPE, EALIGN, ECUDA, ETIMEOUT, EUNSUPPORTED = range(7)

_DTYPE_CODE = {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32,
               torch.uint8: E4M3, torch.float8_e4m3fn: E4M3}
_CODE_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.uint8}

_lock = threading.Lock()
_lib = None
_workspaces = {}


class Fp8LinearError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} (status {status})")


def load():
    """The loaded library (ctypes.CDLL); raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.fp8l_abi_version.restype = I
        lib.fp8l_abi_version.argtypes = []
        version = lib.fp8l_abi_version()
        if version != ABI_VERSION:
            raise RuntimeError(
                f"{LIB_PATH} has ABI version {version}, this binding needs {ABI_VERSION}: "
                f"rebuild it with `python -c \"import __graft_entry__ as g; g.build()\"`")
        lib.fp8l_workspace_bytes.restype = ctypes.c_size_t
        lib.fp8l_workspace_bytes.argtypes = []
        lib.fp8l_strerror.restype = ctypes.c_char_p
        lib.fp8l_strerror.argtypes = [I]
        lib.fp8l_read_status.restype = I
        lib.fp8l_read_status.argtypes = [P, P]
        lib.fp8l_debug_waits.restype = I
        lib.fp8l_debug_waits.argtypes = [ctypes.c_longlong, ctypes.c_uint]
        lib.fp8_quant_per_tensor.restype = I
        lib.fp8_quant_per_tensor.argtypes = [P, I, I64, I64, P, P, I, P, P]
        lib.fp8_quant_per_row.restype = I
        lib.fp8_quant_per_row.argtypes = [P, I, I64, I64, P, P, P]
        lib.fp8_scaled_mm.restype = I
        lib.fp8_scaled_mm.argtypes = [P, P, I64, I64, I64, P, P, I, P, P, I, P, ctypes.c_uint, P]
        lib.fp8_quant_scaled_mm.restype = I
        lib.fp8_quant_scaled_mm.argtypes = [P, I, P, I64, I64, I64, P, I, P, I, P, P, I, P,
                                            ctypes.c_uint, P]
        lib.fp8_quant_scaled_mm_preferred.restype = I
        lib.fp8_quant_scaled_mm_preferred.argtypes = [I64, I64, I64, I]
        lib.fp8_w8a16_mm_kernel.restype = ctypes.c_uint
        lib.fp8_w8a16_mm_kernel.argtypes = [I64, I64, I64, ctypes.c_uint]
        lib.fp8_scaled_mm_kernel.restype = ctypes.c_uint
        lib.fp8_scaled_mm_kernel.argtypes = [I64, I64, I64, ctypes.c_uint]
        lib.fp8_w8a16_mm.restype = I
        lib.fp8_w8a16_mm.argtypes = [P, I, P, P, I64, I64, I64, P, ctypes.c_uint, P]
        lib.fp8_packed_weight_bytes.restype = ctypes.c_size_t
        lib.fp8_packed_weight_bytes.argtypes = [I64, I64]
        lib.fp8_pack_w8a16_weights.restype = I
        lib.fp8_pack_w8a16_weights.argtypes = [P, I64, I64, P, P]
        lib.fp8_grouped_mm.restype = I
        lib.fp8_grouped_mm.argtypes = [P, P, P, I64, I64, I64, I64, P, P, I, P, P, I, P,
                                       ctypes.c_uint, P]
        lib.fp8_rmsnorm_quant.restype = I
        lib.fp8_rmsnorm_quant.argtypes = [P, I, P, ctypes.c_float, I64, I64, P, P, I, P, P, P]
        _lib = lib
        return lib


def strerror(status: int) -> str:
    return load().fp8l_strerror(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise Fp8LinearError(status, where)


def _codes(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not isinstance(t, torch.Tensor) or not t.is_cuda):
            raise TypeError("expected CUDA tensors")
        if t is not None and not t.is_contiguous():
            raise ValueError("expected contiguous tensors")


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def fp8l_workspace_bytes() -> int:
    return int(load().fp8l_workspace_bytes())


def workspace(device=None) -> torch.Tensor:
    """A zero-filled workspace for `device`, allocated once and reused."""
    device = torch.device("cuda", torch.cuda.current_device() if device is None
                          else torch.device(device).index or 0)
    ws = _workspaces.get(device)
    if ws is None:
        ws = torch.zeros(fp8l_workspace_bytes(), dtype=torch.uint8, device=device)
        _workspaces[device] = ws
    return ws


def fp8l_read_status(ws: torch.Tensor) -> int:
    with torch.cuda.device(ws.device):
        return int(load().fp8l_read_status(ws.data_ptr(), _stream(ws.device)))


STALL_MMA = 1
STALL_GRID = 2


def fp8l_debug_waits(wait_cycles: int = 0, stall_mask: int = 0) -> None:
    """Testing hook: shorten the device-side wait limit (cycles; 0 = default)
    and make the given waits target a barrier that nothing completes
    (STALL_MMA, STALL_GRID).  Process-wide; fp8l_debug_waits() restores the
    defaults."""
    _check(load().fp8l_debug_waits(int(wait_cycles), int(stall_mask)), "fp8l_debug_waits")


def fp8_quant_per_tensor(x: torch.Tensor, q: torch.Tensor | None = None,
                         scale: torch.Tensor | None = None, dynamic: bool = True,
                         ws: torch.Tensor | None = None):
    """Per-tensor E4M3 quantization of x.  Returns (q uint8, scale float32[1]).
    dynamic=False reads the given `scale` (static input scale)."""
    _need_cuda(x, q, scale, ws)
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        if not dynamic:
            raise ValueError("static quantization needs a scale tensor")
        scale = torch.empty(1, dtype=torch.float32, device=x.device)
    if dynamic and ws is None:
        ws = workspace(x.device)
    rows = x.shape[0] if x.dim() > 1 else 1
    cols = x.numel() // rows if rows else 0
    with torch.cuda.device(x.device):
        st = load().fp8_quant_per_tensor(
            x.data_ptr(), _DTYPE_CODE[x.dtype], rows, cols, _codes(q).data_ptr(),
            scale.data_ptr(), 1 if dynamic else 0, ws.data_ptr() if ws is not None else None,
            _stream(x.device))
    _check(st, "fp8_quant_per_tensor")
    return q, scale


NQ_MODES = {"dynamic": 0, "static": 1, "per_token": 2, "norm_only": 3}


def fp8_rmsnorm_quant(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-5,
                      mode: str = "dynamic", q: torch.Tensor | None = None,
                      scale: torch.Tensor | None = None, h: torch.Tensor | None = None,
                      want_h: bool = False, ws: torch.Tensor | None = None):
    """RMSNorm of x [M, K] (fp16/bf16) with gamma [K], fused with its E4M3
    quantization.  mode: "dynamic" (per-tensor scale written), "static"
    (scale given), "per_token" (M scales written) or "norm_only" (h only).
    Returns (q uint8 or None, scale or None, h or None); h is written when
    given, when want_h, or in norm_only mode."""
    _need_cuda(x, gamma, q, scale, h, ws)
    if x.dim() != 2 or gamma.shape != (x.shape[1],) or gamma.dtype != x.dtype:
        raise ValueError("expected x [M, K] and gamma [K] of the same dtype")
    M, K = x.shape
    m = NQ_MODES[mode]
    if (want_h or mode == "norm_only") and h is None:
        h = torch.empty_like(x)
    if mode != "norm_only":
        if q is None:
            q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
        if scale is None:
            if mode == "static":
                raise ValueError("static mode needs a scale tensor")
            scale = torch.empty(M if mode == "per_token" else 1, dtype=torch.float32,
                                device=x.device)
    if mode == "dynamic" and ws is None:
        ws = workspace(x.device)
    with torch.cuda.device(x.device):
        st = load().fp8_rmsnorm_quant(
            x.data_ptr(), _DTYPE_CODE[x.dtype], gamma.data_ptr(), float(eps), M, K,
            _codes(q).data_ptr() if q is not None else None,
            scale.data_ptr() if scale is not None else None, m,
            h.data_ptr() if h is not None else None,
            ws.data_ptr() if ws is not None else None, _stream(x.device))
    _check(st, "fp8_rmsnorm_quant")
    return q, scale, h


def fp8_quant_per_row(x: torch.Tensor, q: torch.Tensor | None = None,
                      row_scale: torch.Tensor | None = None):
    """One dynamic scale per row of a 2-D tensor.  Returns (q uint8, scales float32[rows])."""
    _need_cuda(x, q, row_scale)
    if x.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if row_scale is None:
        row_scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        st = load().fp8_quant_per_row(x.data_ptr(), _DTYPE_CODE[x.dtype], rows, cols,
                                      _codes(q).data_ptr(), row_scale.data_ptr(),
                                      _stream(x.device))
    _check(st, "fp8_quant_per_row")
    return q, row_scale


def scaled_mm_kernel(M: int, N: int, K: int, kernel: str = "auto") -> str:
    """Name ("stream", "swapped" or "tiled") of the kernel fp8_scaled_mm runs
    for this shape and kernel choice (fp8_scaled_mm_kernel; no GPU needed)."""
    code = load().fp8_scaled_mm_kernel(M, N, K, KERNELS[kernel])
    return {v: k for k, v in KERNELS.items()}[code]


def quant_scaled_mm_preferred(M: int, N: int, K: int, dynamic: bool = True) -> bool:
    """Whether fp8_quant_scaled_mm takes this shape and is the faster way to
    run it (fp8_quant_scaled_mm_preferred; no GPU needed)."""
    return bool(load().fp8_quant_scaled_mm_preferred(M, N, K, 1 if dynamic else 0))


def fp8_quant_scaled_mm(x: torch.Tensor, w: torch.Tensor, w_scale: torch.Tensor,
                        a_scale: torch.Tensor | None = None, dynamic: bool = True,
                        out_dtype=torch.bfloat16, out_scale: torch.Tensor | None = None,
                        y: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                        stable_weights: bool = False, kernel: str = "auto"):
    """W8A8 product of 16-bit x [M <= 128, K] and E4M3 w [N, K] with the
    per-tensor activation quantization fused into it (fp8_quant_scaled_mm):
    dynamic writes a_scale (a new [1] tensor when None), static reads it.
    kernel: "auto" (the one fp8_scaled_mm would run, tiles excepted),
    "stream" (up to 16 tokens) or "swapped".  Returns (y, a_scale)."""
    _need_cuda(x, w, w_scale, a_scale, out_scale, y, ws)
    w = _codes(w)
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("inner dimensions differ")
    if a_scale is None:
        if not dynamic:
            raise ValueError("a static scale must be given")
        a_scale = torch.empty(1, dtype=torch.float32, device=x.device)
    if out_dtype == torch.float8_e4m3fn:
        out_dtype = torch.uint8
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if ws is None:
        ws = workspace(x.device)
    if w_scale.numel() not in (1, N):
        raise ValueError("w_scale must have 1 or N entries")
    per_channel = 1 if w_scale.numel() == N and N != 1 else 0
    with torch.cuda.device(x.device):
        st = load().fp8_quant_scaled_mm(
            x.data_ptr(), _DTYPE_CODE[x.dtype], w.data_ptr(), M, N, K, a_scale.data_ptr(),
            1 if dynamic else 0, w_scale.data_ptr(), per_channel,
            out_scale.data_ptr() if out_scale is not None else None, _codes(y).data_ptr(),
            _DTYPE_CODE[y.dtype], ws.data_ptr(),
            (WEIGHTS_STABLE if stable_weights else 0) | KERNELS[kernel], _stream(x.device))
    _check(st, "fp8_quant_scaled_mm")
    return y, a_scale


def w8a16_mm_kernel(M: int, N: int, K: int, kernel: str = "auto") -> str:
    """Name ("stream" or "swapped") of the kernel fp8_w8a16_mm runs for this
    shape and kernel choice (fp8_w8a16_mm_kernel; no GPU needed)."""
    code = load().fp8_w8a16_mm_kernel(M, N, K, KERNELS[kernel])
    return {v: k for k, v in KERNELS.items()}[code]


def fp8_scaled_mm(a: torch.Tensor, w: torch.Tensor, a_scale: torch.Tensor,
                  w_scale: torch.Tensor, out_dtype=torch.bfloat16,
                  out_scale: torch.Tensor | None = None, y: torch.Tensor | None = None,
                  ws: torch.Tensor | None = None, stable_weights: bool = False,
                  per_token: bool | None = None, single_sm: bool = False,
                  kernel: str = "auto") -> torch.Tensor:
    """W8A8 product of E4M3 a [M, K] and w [N, K] with a per-tensor ([1]) or
    per-token ([M]) a_scale and a per-tensor ([1]) or per-channel ([N])
    w_scale.  out_dtype bf16 / fp16, or uint8 (E4M3 codes, needs out_scale).
    stable_weights sets FP8L_WEIGHTS_STABLE (no work in flight on the stream
    writes w or w_scale); per_token (default: a_scale has M > 1 entries) sets
    FP8L_A_PER_TOKEN; single_sm sets FP8L_SINGLE_SM_TILES; kernel ("auto",
    "stream", "swapped" or "tiled") sets the FP8L_KERNEL_* choice."""
    _need_cuda(a, w, a_scale, w_scale, out_scale, y, ws)
    a, w = _codes(a), _codes(w)
    M, K = a.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("inner dimensions differ")
    if out_dtype == torch.float8_e4m3fn:
        out_dtype = torch.uint8
    code = _DTYPE_CODE[out_dtype]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=a.device)
    if ws is None:
        ws = workspace(a.device)
    per_channel = 1 if w_scale.numel() == N and N != 1 else 0
    if w_scale.numel() not in (1, N):
        raise ValueError("w_scale must have 1 or N entries")
    if per_token is None:
        per_token = a_scale.numel() == M and M > 1
    if a_scale.numel() != (M if per_token else 1):
        raise ValueError("a_scale must have 1 entry, or M with per_token")
    flags = ((WEIGHTS_STABLE if stable_weights else 0) | (A_PER_TOKEN if per_token else 0) |
             (SINGLE_SM_TILES if single_sm else 0) | KERNELS[kernel])
    with torch.cuda.device(a.device):
        st = load().fp8_scaled_mm(
            a.data_ptr(), w.data_ptr(), M, N, K, a_scale.data_ptr(), w_scale.data_ptr(),
            per_channel, out_scale.data_ptr() if out_scale is not None else None,
            _codes(y).data_ptr(), code, ws.data_ptr(), flags, _stream(a.device))
    _check(st, "fp8_scaled_mm")
    return y


def fp8_grouped_mm(a: torch.Tensor, w: torch.Tensor, group_offsets: torch.Tensor,
                   a_scale: torch.Tensor, w_scale: torch.Tensor, out_dtype=torch.bfloat16,
                   out_scale: torch.Tensor | None = None, y: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None, stable_weights: bool = False,
                   per_token: bool | None = None) -> torch.Tensor:
    """Grouped W8A8 product of mixture-of-experts layers: rows
    group_offsets[e] .. group_offsets[e+1]-1 of E4M3 a [M, K] times expert
    e's E4M3 weights w[e] [N, K].  group_offsets: int32 [E + 1] on the
    device; w_scale: [E] (per expert) or [E, N] (per channel); a_scale [1] or
    [M] (per token).  Rows outside the groups of a freshly allocated y are
    zero-filled first; a given y keeps them."""
    _need_cuda(a, w, group_offsets, a_scale, w_scale, out_scale, y, ws)
    a, w = _codes(a), _codes(w)
    M, K = a.shape
    E, N, K2 = w.shape
    if K2 != K or group_offsets.numel() != E + 1 or group_offsets.dtype != torch.int32:
        raise ValueError("shape mismatch")
    per_channel = w_scale.numel() == E * N and N != 1
    if w_scale.numel() not in (E, E * N):
        raise ValueError("w_scale must have E or E * N entries")
    if per_token is None:
        per_token = a_scale.numel() == M and M > 1
    if out_dtype == torch.float8_e4m3fn:
        out_dtype = torch.uint8
    if y is None:
        y = torch.zeros((M, N), dtype=out_dtype, device=a.device)
    if ws is None:
        ws = workspace(a.device)
    flags = (WEIGHTS_STABLE if stable_weights else 0) | (A_PER_TOKEN if per_token else 0)
    with torch.cuda.device(a.device):
        st = load().fp8_grouped_mm(
            a.data_ptr(), w.data_ptr(), group_offsets.data_ptr(), E, M, N, K,
            a_scale.data_ptr(), w_scale.data_ptr(), 1 if per_channel else 0,
            out_scale.data_ptr() if out_scale is not None else None, _codes(y).data_ptr(),
            _DTYPE_CODE[y.dtype], ws.data_ptr(), flags, _stream(a.device))
    _check(st, "fp8_grouped_mm")
    return y


def fp8_packed_weight_bytes(N: int, K: int) -> int:
    """Bytes of the packed layout of [N, K] E4M3 weights (0 for a bad shape)."""
    return int(load().fp8_packed_weight_bytes(N, K))


def fp8_pack_w8a16_weights(w: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """The packed copy of E4M3 weight codes w [N, K] that fp8_w8a16_mm reads
    with packed=True: a 1-D uint8 tensor of fp8_packed_weight_bytes(N, K)."""
    _need_cuda(w, out)
    w = _codes(w)
    N, K = w.shape
    nbytes = fp8_packed_weight_bytes(N, K)
    if nbytes == 0:
        _check(ESHAPE, "fp8_pack_w8a16_weights")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    elif out.dtype != torch.uint8 or out.numel() != nbytes:
        raise ValueError("out must be a uint8 tensor of fp8_packed_weight_bytes(N, K) elements")
    with torch.cuda.device(w.device):
        st = load().fp8_pack_w8a16_weights(w.data_ptr(), N, K, out.data_ptr(), _stream(w.device))
    _check(st, "fp8_pack_w8a16_weights")
    return out


def fp8_w8a16_mm(x: torch.Tensor, w: torch.Tensor, w_scale: torch.Tensor,
                 y: torch.Tensor | None = None, stable_weights: bool = False,
                 packed: bool = False, kernel: str = "auto") -> torch.Tensor:
    """Weight-only product: fp16/bf16 x [M, K] times E4M3 w [N, K] with
    per-channel w_scale [N]; the output has x's dtype.  stable_weights sets
    FP8L_WEIGHTS_STABLE (no work in flight on the stream writes w or
    w_scale).  packed: w is the output of fp8_pack_w8a16_weights (N is
    taken from w_scale) and FP8L_WEIGHTS_PACKED is set.  kernel ("auto",
    "stream" or "swapped") sets the FP8L_KERNEL_* choice."""
    _need_cuda(x, w, w_scale, y)
    w = _codes(w)
    M, K = x.shape
    N = w_scale.numel()
    if packed:
        if w.dtype != torch.uint8 or w.numel() != fp8_packed_weight_bytes(N, K):
            raise ValueError("packed weights must be fp8_pack_w8a16_weights output for [N, K]")
    elif w.dim() != 2 or w.shape[0] != N or w.shape[1] != K:
        raise ValueError("shape mismatch")
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    flags = ((WEIGHTS_STABLE if stable_weights else 0) | (WEIGHTS_PACKED if packed else 0) |
             KERNELS[kernel])
    with torch.cuda.device(x.device):
        st = load().fp8_w8a16_mm(x.data_ptr(), _DTYPE_CODE[x.dtype], w.data_ptr(),
                                 w_scale.data_ptr(), M, N, K, y.data_ptr(), flags,
                                 _stream(x.device))
    _check(st, "fp8_w8a16_mm")
    return y
