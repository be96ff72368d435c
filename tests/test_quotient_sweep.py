"""The quantizer kernels form RN(x / s) without a per-element division: a
product with the correctly rounded reciprocal and fused multiply-add
corrections (one for 16-bit inputs, two for fp32; Markstein's theorem, P.
Markstein, IBM J. Res. Develop. 34(1), 1990, gives the fp32 case).  The
claim that one correction already gives the IEEE quotient for 16-bit inputs
rests on an exhaustive check, replayed here on the host with the C library's
correctly rounded fmaf: every (bfloat16 significand, fp32 significand) pair,
2^30 pairs; fp16 on a regular sample of 2^27 pairs.  A single product
without correction fails, which shows the sweep can see a difference.

This compares the kernels' method with IEEE division (the oracle's
definition of the quotient); the GPU tests then compare the kernels' codes
with the oracle's over every 16-bit value and hundreds of scales."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def sweep(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("qs") / "libqs.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
                    "-fPIC", "-shared", os.path.join(HERE, "quotient_sweep.c"), "-o", out,
                    "-lm"], check=True)
    lib = ctypes.CDLL(out)
    lib.qs_sweep16.restype = ctypes.c_int64
    lib.qs_sweep16.argtypes = [ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                               ctypes.c_int, ctypes.POINTER(ctypes.c_uint32),
                               ctypes.POINTER(ctypes.c_uint32)]
    lib.qs_pairs.restype = ctypes.c_int64
    lib.qs_pairs.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
    return lib


def _run(lib, x_bits, s_lo, s_hi, step, corrections):
    bx, bs = ctypes.c_uint32(), ctypes.c_uint32()
    bad = lib.qs_sweep16(x_bits, s_lo, s_hi, step, corrections, ctypes.byref(bx),
                         ctypes.byref(bs))
    return bad, hex(bx.value), hex(bs.value)


def test_bfloat16_one_correction_exhaustive(sweep):
    bad = _run(sweep, 7, 0, 1 << 23, 1, 1)
    assert bad[0] == 0, bad


def test_fp16_one_correction_sampled(sweep):
    # every fp16 significand against every 64th fp32 significand (all 2^17
    # of them share no structure with the stride), 2^27 pairs
    bad = _run(sweep, 10, 0, 1 << 23, 64, 1)
    assert bad[0] == 0, bad
    bad = _run(sweep, 10, 37, 1 << 23, 64, 1)
    assert bad[0] == 0, bad


def test_the_sweep_sees_an_uncorrected_product(sweep):
    bad = _run(sweep, 7, 0, 1 << 16, 1, 0)
    assert bad[0] > 0


def test_fp32_two_corrections_random_pairs(sweep):
    rng = np.random.default_rng(8)
    n = 1 << 24
    # significands over [1, 2) and exponents spread so quotients cover
    # (0.5, 2) times powers of two well inside the normal range
    mx = rng.integers(0, 1 << 23, n, dtype=np.uint32)
    ms = rng.integers(0, 1 << 23, n, dtype=np.uint32)
    ex = rng.integers(-20, 21, n).astype(np.int64)
    es = rng.integers(-20, 21, n).astype(np.int64)
    x = (((127 + ex) << 23).astype(np.uint32) | mx).astype(np.uint32)
    s = (((127 + es) << 23).astype(np.uint32) | ms).astype(np.uint32)
    assert sweep.qs_pairs(x.ctypes.data, s.ctypes.data, n, 2) == 0
    # and the check sees the uncorrected product differ
    assert sweep.qs_pairs(x.ctypes.data, s.ctypes.data, n, 0) > 0
