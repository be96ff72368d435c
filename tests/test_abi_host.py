"""Host-side checks of the C ABI: the library builds, loads without a GPU,
exports every entry point the header declares, and rejects bad arguments
before touching CUDA.  No kernel is launched here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8linear.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_quantized_linear_gb300 import build
    build.build()
    import fp8_quantized_linear_gb300 as fl
    return fl.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fp8\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("fp8_quant_per_tensor", "fp8_quant_per_row", "fp8_scaled_mm", "fp8_w8a16_mm",
                 "fp8_pack_w8a16_weights", "fp8_packed_weight_bytes",
                 "fp8l_workspace_bytes", "fp8l_read_status", "fp8l_strerror", "fp8l_abi_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from fp8_quantized_linear_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_only_c_abi_symbols_exported(lib):
    from fp8_quantized_linear_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert all(n.startswith("fp8") for n in exported), sorted(n for n in exported if not n.startswith("fp8"))


def test_constants(lib):
    import fp8_quantized_linear_gb300 as fl
    assert lib.fp8l_abi_version() == fl._binding.ABI_VERSION == 7
    assert fl.fp8l_workspace_bytes() >= 4096 and fl.fp8l_workspace_bytes() % 16 == 0
    for code in range(7):
        assert fl.strerror(code)
    assert "unknown" in fl.strerror(99)


P = ctypes.c_void_p
A16 = 0x10000  # a fake, 16-byte aligned address: never dereferenced


def test_scaled_mm_argument_errors(lib):
    import fp8_quantized_linear_gb300._binding as b
    f = lib.fp8_scaled_mm
    ok = dict(a=A16, w=A16, M=32, N=32, K=32, sa=A16, sw=A16, pc=0, os=None, y=A16,
              od=b.BF16, ws=A16, fl=0, st=None)

    def call(**kw):
        d = dict(ok)
        d.update(kw)
        return f(d["a"], d["w"], d["M"], d["N"], d["K"], d["sa"], d["sw"], d["pc"], d["os"],
                 d["y"], d["od"], d["ws"], d["fl"], d["st"])
    assert call(od=7) == b.EINVAL
    assert call(sa=None) == b.EINVAL
    assert call(w=None) == b.EINVAL
    assert call(ws=None) == b.EINVAL
    assert call(od=b.E4M3, os=None) == b.EINVAL
    assert call(N=24) == b.ESHAPE
    assert call(K=8) == b.ESHAPE
    assert call(K=0) == b.ESHAPE
    assert call(M=-1) == b.ESHAPE
    assert call(N=(1 << 20) + 16) == b.ESHAPE
    assert call(a=None) == b.EINVAL
    assert call(a=A16 + 8) == b.EALIGN
    assert call(y=A16 + 4) == b.EALIGN
    assert call(sw=A16 + 2) == b.EALIGN
    assert call(fl=2) == b.EINVAL
    assert call(fl=64) == b.EINVAL
    assert call(fl=b.KERNELS["swapped"], M=129) == b.ESHAPE


def test_scaled_mm_kernel_choice(lib):
    # which kernel fp8_scaled_mm runs: a pure function of the shape, no GPU
    import fp8_quantized_linear_gb300 as fl
    k = fl.scaled_mm_kernel
    assert k(16, 256, 512) == "stream"        # tiny layer
    assert k(1, 4096, 4096) == "stream"       # 16 MiB of weights
    assert k(16, 4096, 4096) == "stream"
    assert k(4, 6144, 4096) == "stream"       # 24 MiB at up to 4 tokens
    assert k(16, 6144, 4096) == "swapped"
    assert k(1, 28672, 4096) == "swapped"
    assert k(64, 10240, 8192) == "swapped"
    assert k(128, 4096, 14336) == "swapped"
    assert k(128, 57344, 8192) == "tiled"     # 448 MiB above 64 tokens
    assert k(64, 57344, 8192) == "swapped"
    assert k(129, 4096, 4096) == "tiled"
    assert k(1024, 4096, 4096) == "tiled"
    for name in ("stream", "swapped", "tiled"):  # an explicit choice is kept
        assert k(1024, 4096, 4096, name) == name


def test_quant_scaled_mm_preferred(lib):
    # when the fused quantization + product is the faster call: a pure
    # function of the shape, no GPU
    import fp8_quantized_linear_gb300 as fl
    p = fl.quant_scaled_mm_preferred
    assert p(1, 28672, 4096)                  # 224 weight blocks, one wave at 8 tokens or fewer
    assert p(8, 28672, 4096, dynamic=False)
    assert p(1, 4096, 14336)                  # dynamic: 28 KB of x
    assert not p(4, 4096, 14336)              # dynamic: 112 KB of x, over the limit
    assert p(4, 4096, 14336, dynamic=False)
    assert p(1, 38912, 4096)                  # 304 blocks
    assert not p(1, 38928, 4096)              # 305 blocks: a second wave
    assert not p(1, 57344, 8192)
    assert p(16, 6144, 4096, dynamic=False)   # 48 blocks: clusters split K
    assert p(16, 19456, 4096, dynamic=False)  # 152 blocks
    assert not p(16, 19472, 4096, dynamic=False)
    assert not p(16, 28672, 4096, dynamic=False)
    assert not p(16, 6144, 4096)              # dynamic: 128 KB of x
    assert not p(17, 6144, 1024, dynamic=False)
    # small weights, the CUDA-core weight stream: one token tile, or short rows
    assert p(8, 4096, 4096, dynamic=False) and p(1, 4096, 4096)
    assert not p(16, 4096, 4096, dynamic=False)
    assert p(16, 256, 512)                    # the tiny layer
    assert not p(0, 4096, 4096) and not p(1, 4100, 4096) and not p(1, 4096, 0)


def test_quant_scaled_mm_argument_errors(lib):
    import fp8_quantized_linear_gb300._binding as b
    f = lib.fp8_quant_scaled_mm
    ok = dict(x=A16, xd=b.BF16, w=A16, M=16, N=32, K=64, sa=A16, dyn=1, sw=A16, pc=0, os=None,
              y=A16, od=b.BF16, ws=A16, fl=0, st=None)

    def call(**kw):
        d = dict(ok)
        d.update(kw)
        return f(d["x"], d["xd"], d["w"], d["M"], d["N"], d["K"], d["sa"], d["dyn"], d["sw"], d["pc"],
                 d["os"], d["y"], d["od"], d["ws"], d["fl"], d["st"])
    assert call(xd=b.E4M3) == b.EINVAL
    assert call(xd=b.F32) == b.EINVAL
    assert call(od=7) == b.EINVAL
    assert call(fl=2) == b.EINVAL
    assert call(sa=None) == b.EINVAL
    assert call(od=b.E4M3, os=None) == b.EINVAL
    assert call(fl=b.KERNELS["tiled"]) == b.EINVAL
    assert call(fl=b.KERNELS["stream"], M=17, dyn=0) == b.ESHAPE
    assert call(M=129) == b.ESHAPE
    assert call(N=24) == b.ESHAPE
    # dynamic: every CTA reads all of x, so x is bounded
    assert call(M=4, K=8192 + 16) == b.ESHAPE
    assert call(x=A16 + 8) == b.EALIGN
    assert call(sa=A16 + 2) == b.EALIGN


def test_w8a16_mm_kernel_choice(lib):
    import fp8_quantized_linear_gb300 as fl
    k = fl.w8a16_mm_kernel
    assert k(1, 4096, 4096) == "stream"
    assert k(8, 22016, 4096) == "stream"
    assert k(16, 12288, 4096) == "stream"
    assert k(17, 4096, 4096) == "swapped"
    assert k(64, 4096, 11008) == "swapped"
    assert k(65, 4096, 4096) == "stream"
    assert k(16, 4096, 4096, "stream") == "stream"
    assert k(1, 4096, 4096, "swapped") == "swapped"


def test_w8a16_argument_errors(lib):
    import fp8_quantized_linear_gb300._binding as b
    f = lib.fp8_w8a16_mm
    assert f(A16, b.E4M3, A16, A16, 1, 32, 32, A16, 0, None) == b.EINVAL
    assert f(A16, b.F32, A16, A16, 1, 32, 32, A16, 0, None) == b.EINVAL
    assert f(A16, b.F16, A16, A16, 1, 32, 32, A16, 6, None) == b.EINVAL
    assert f(A16, b.F16, A16, A16, 1, 40, 32, A16, 0, None) == b.ESHAPE
    assert f(A16, b.F16, A16, A16, 1, 32, 40, A16, 0, None) == b.ESHAPE
    assert f(A16, b.F16, None, A16, 1, 32, 32, A16, 0, None) == b.EINVAL
    assert f(A16 + 2, b.F16, A16, A16, 1, 32, 32, A16, 0, None) == b.EALIGN
    assert f(A16, b.F16, A16, A16, 1, 32, 32, A16, 4, None) == b.EINVAL
    assert f(A16, b.F16, A16, A16, 1, 32, 32, A16, b.WEIGHTS_PACKED | 8, None) == b.EINVAL
    assert f(A16, b.F16, A16, A16, 1, 32, 32, A16, b.KERNELS["tiled"], None) == b.EINVAL
    assert f(A16, b.F16, A16, A16, 65, 32, 32, A16, b.KERNELS["swapped"], None) == b.ESHAPE


def test_packed_weight_bytes_and_pack_argument_errors(lib):
    import fp8_quantized_linear_gb300._binding as b
    nb = lib.fp8_packed_weight_bytes
    # N rows of ceil(K / 64) 64-byte chunks
    assert nb(32, 4096) == 32 * 4096
    assert nb(32, 208) == 32 * 256
    assert nb(16, 16) == 16 * 64
    assert nb(4096, 11008) == 4096 * 11008
    for n, k in ((24, 64), (32, 0), (-16, 32), (32, 40), ((1 << 20) + 16, 64), (16, 1 << 21)):
        assert nb(n, k) == 0, (n, k)
    f = lib.fp8_pack_w8a16_weights
    assert f(A16, 24, 64, A16, None) == b.ESHAPE
    assert f(A16, 32, 40, A16, None) == b.ESHAPE
    assert f(None, 32, 64, A16, None) == b.EINVAL
    assert f(A16, 32, 64, None, None) == b.EINVAL
    assert f(A16 + 8, 32, 64, A16, None) == b.EALIGN
    assert f(A16, 32, 64, A16 + 4, None) == b.EALIGN


def test_quant_argument_errors(lib):
    import fp8_quantized_linear_gb300._binding as b
    f = lib.fp8_quant_per_tensor
    assert f(A16, b.E4M3, 4, 4, A16, A16, 1, A16, None) == b.EINVAL
    assert f(A16, b.BF16, 4, 4, A16, None, 1, A16, None) == b.EINVAL
    assert f(A16, b.BF16, 4, 4, A16, A16, 1, None, None) == b.EINVAL
    assert f(A16, b.BF16, -1, 4, A16, A16, 1, A16, None) == b.ESHAPE
    assert f(A16, b.BF16, 1 << 30, 1 << 20, A16, A16, 1, A16, None) == b.ESHAPE
    assert f(A16 + 8, b.BF16, 4, 4, A16, A16, 1, A16, None) == b.EALIGN
    assert f(A16, b.BF16, 4, 4, A16, A16 + 1, 1, A16, None) == b.EALIGN
    g = lib.fp8_quant_per_row
    assert g(A16, b.BF16, 4, 24, A16, A16, None) == b.ESHAPE
    assert g(A16, 9, 4, 32, A16, A16, None) == b.EINVAL
    assert g(A16, b.BF16, 4, 32, None, A16, None) == b.EINVAL


def test_debug_waits_argument_errors(lib):
    import fp8_quantized_linear_gb300._binding as b
    lib.fp8l_debug_waits.restype = ctypes.c_int
    lib.fp8l_debug_waits.argtypes = [ctypes.c_longlong, ctypes.c_uint]
    assert lib.fp8l_debug_waits(-1, 0) == b.EINVAL
    assert lib.fp8l_debug_waits(0, 4) == b.EINVAL
    assert lib.fp8l_debug_waits(1 << 20, b.STALL_MMA | b.STALL_GRID) == b.OK
    assert lib.fp8l_debug_waits(0, 0) == b.OK  # back to the defaults


def test_read_status_argument_errors(lib):
    import fp8_quantized_linear_gb300._binding as b
    assert lib.fp8l_read_status(None, None) == b.EINVAL
    assert lib.fp8l_read_status(A16 + 4, None) == b.EALIGN


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import fp8_quantized_linear_gb300._binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        b.load()


def test_library_of_another_abi_version_is_refused(monkeypatch, tmp_path):
    import fp8_quantized_linear_gb300._binding as b
    stale = tmp_path / "libfp8linear.so"
    stale.write_bytes(b"")

    class OldLib:
        class _Fn:
            restype = None
            argtypes = None

            def __call__(self):
                return 1

        fp8l_abi_version = _Fn()

    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(stale))
    monkeypatch.setattr(b.ctypes, "CDLL", lambda path: OldLib())
    with pytest.raises(RuntimeError, match="ABI version 1"):
        b.load()


def test_cpu_tensors_are_refused_not_computed():
    # there is no CPU fallback: every entry point wants CUDA tensors
    import torch
    import fp8_quantized_linear_gb300 as fl
    x = torch.zeros((4, 32), dtype=torch.bfloat16)
    q = torch.zeros((32, 32), dtype=torch.uint8)
    one = torch.ones(1)
    calls = [
        lambda: fl.fp8_quant_per_tensor(x),
        lambda: fl.fp8_quant_per_row(x),
        lambda: fl.fp8_scaled_mm(q, q, one, one),
        lambda: fl.fp8_w8a16_mm(x.half(), q, torch.ones(32)),
        lambda: fl.fp8_pack_w8a16_weights(q),
    ]
    for call in calls:
        with pytest.raises(TypeError, match="CUDA"):
            call()


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "fp8_quantized_linear_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"\boracle\b", text), os.path.join(dirpath, fn)
                assert "fp8_oracle" not in text
