"""Pins: checks that tie an implementation of the layer's arithmetic to facts
fixed outside it (hand-derived golden values, closed forms, invariants,
library casts, exact integer arithmetic).

Each check takes the implementation under test as an argument, so the same
checks run on the CPU oracle (test_oracle_*.py) and on deliberately broken
copies of it (test_oracle_mutants.py), which shows that each kind of plausible
mistake is caught.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _strip(line):
    return line.split("#", 1)[0].strip()


def load_landmarks():
    out = []
    with open(os.path.join(GOLDEN, "e4m3_landmarks.txt")) as f:
        for line in f:
            line = _strip(line)
            if line:
                code, val = line.split()
                out.append((int(code, 16), float(val)))
    return out


def load_rounding():
    out = []
    with open(os.path.join(GOLDEN, "e4m3_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            out.append((float(parts[0]), int(parts[1], 16)))
    return out


def load_worked_quant():
    cases = []
    with open(os.path.join(GOLDEN, "quant_per_tensor_worked.txt")) as f:
        for line in f:
            line = _strip(line)
            if not line:
                continue
            lhs, rhs = line.split(";")
            parts = lhs.split()
            name, sbits, xs = parts[0], int(parts[1], 16), [float(v) for v in parts[2:]]
            codes = [int(c, 16) for c in rhs.split()]
            cases.append((name, sbits, xs, codes))
    return cases


# ---------------------------------------------------------------------------
# library casts (the special case "clamp to the finite range, then the
# library's round-to-nearest-even cast" equals the saturating cast)

def torch_e4m3_codes(values_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(values_f32, dtype=np.float32))
    return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def all_16bit_values(dtype) -> np.ndarray:
    """Every finite value of a 16-bit float format, as float32."""
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    vals = bits.view(dtype).float()
    vals = vals[torch.isfinite(vals)]
    return vals.numpy()


# ---------------------------------------------------------------------------
# E4M3 decode

def check_decode_table(table: np.ndarray):
    assert table.shape == (256,)
    for code, val in load_landmarks():
        got = table[code]
        if math.isnan(val):
            assert math.isnan(got), (hex(code), got)
        else:
            assert got == val, (hex(code), got, val)
            assert math.copysign(1.0, got) == math.copysign(1.0, val), hex(code)
    # library decode of every code
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(table), nan)
    assert np.array_equal(table[~nan], lib[~nan])
    assert np.array_equal(np.signbit(table[~nan]), np.signbit(lib[~nan]))
    # 127 strictly increasing non-negative finite values, mirrored by sign
    pos = table[:127]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(table[128:255], -pos)


# ---------------------------------------------------------------------------
# E4M3 encode: ``encode(values float64 array) -> uint8 codes``

def check_encoder(encode, table: np.ndarray):
    vals = np.array([v for v, _ in load_rounding()], dtype=np.float64)
    want = np.array([c for _, c in load_rounding()], dtype=np.uint8)
    got = encode(vals)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(vals[i], hex(got[i]), hex(want[i])) for i in bad]
    # every finite code is the encoding of its own value
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    rt = encode(table[finite])
    assert np.array_equal(rt, finite.astype(np.uint8))
    # agreement with the library cast on every bf16 and fp16 value
    for dt in (torch.bfloat16, torch.float16):
        v = all_16bit_values(dt)
        got = encode(v.astype(np.float64))
        lib = torch_e4m3_codes(v)
        bad = np.nonzero(got != lib)[0]
        assert bad.size == 0, (dt, [(v[i], hex(got[i]), hex(lib[i])) for i in bad[:8]])
    # and on random float32 values over the whole useful range
    rng = np.random.default_rng(1234)
    v = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-14, 10, 200_000))).astype(np.float32)
    got = encode(v.astype(np.float64))
    assert np.array_equal(got, torch_e4m3_codes(v))


def linear_scan_encode(v: float, table: np.ndarray) -> int:
    """Independent restatement for brute-force spot checks: scan every finite
    non-negative code for the nearest value, ties to the even code."""
    if math.isnan(v):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a >= 448.0:
        return sign | 0x7E
    best, bestd = None, None
    for c in range(127):
        d = abs(table[c] - a)
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return sign | best


# ---------------------------------------------------------------------------
# per-tensor quantization: ``quant(x_torch, scale=None) -> (codes, scale)``

def check_quant_worked(quant):
    for name, sbits, xs, codes in load_worked_quant():
        for dt in (torch.bfloat16, torch.float16, torch.float32):
            x = torch.tensor(xs, dtype=torch.float32).to(dt)
            assert x.float().tolist() == xs, (name, dt)  # inputs are exact
            q, s = quant(x)
            assert int(np.float32(s).view(np.uint32)) == sbits, (name, dt, hex(int(np.float32(s).view(np.uint32))))
            assert list(np.asarray(q).reshape(-1)) == codes, (name, dt, [hex(c) for c in np.asarray(q).reshape(-1)])


def check_quant_invariants(quant, table: np.ndarray, x: torch.Tensor):
    xf = x.float().numpy().reshape(-1)
    q, s = quant(x)
    q = np.asarray(q).reshape(-1)
    s = np.float32(s)
    amax = np.abs(xf).max()
    assert s > 0
    # no NaN codes; every |value| <= 448
    assert not np.any((q & 0x7F) == 0x7F)
    dec = table[q]
    assert np.all(np.abs(dec) <= 448.0)
    if amax > 0:
        # the element of largest magnitude lands on +-448
        i = int(np.argmax(np.abs(xf)))
        assert (q[i] & 0x7F) == 0x7E, (hex(q[i]), amax, s)
        # half-spacing error bound, normal and subnormal range of E4M3
        err = np.abs(dec * np.float64(s) - xf.astype(np.float64))
        bound = np.maximum(np.abs(xf.astype(np.float64)) * 2.0 ** -4, np.float64(s) * 2.0 ** -10)
        assert np.all(err <= bound * (1 + 4e-6)), float(np.max(err / bound))
        # sign is kept
        nz = dec != 0
        assert np.all(np.sign(dec[nz]) == np.sign(xf[nz]))
    else:
        assert s == np.float32(1.0)
        assert np.all((q & 0x7F) == 0)
    # monotone: x_i <= x_j implies dec(q_i) <= dec(q_j)
    order = np.argsort(xf, kind="stable")
    assert np.all(np.diff(dec[order]) >= 0)
    # power-of-two equivariance (no over/underflow for these inputs)
    for k in ((-3, 5) if amax > 0 else ()):
        q2, s2 = quant((x.float() * 2.0 ** k).to(x.dtype))
        assert np.float32(s2) == np.float32(s * np.float32(2.0 ** k))
        assert np.array_equal(np.asarray(q2).reshape(-1), q)


def check_quant_static(quant, encode):
    x = torch.tensor([0.1, -0.7, 3.0, 1000.0, -1e-6], dtype=torch.float32)
    s = np.float32(0.0123)
    q, s_out = quant(x, scale=s)
    assert np.float32(s_out) == s
    want = encode((x.numpy() / s).astype(np.float32).astype(np.float64))
    assert np.array_equal(np.asarray(q).reshape(-1), want)
    assert q[3] == 0x7E  # 1000/0.0123 saturates


# ---------------------------------------------------------------------------
# W8A8 scaled product: ``mm(qa, qw, sa, sw) -> y float64 [M, N]``

def _code_of(table, v):
    return int(np.nonzero(table == v)[0][0])


def check_scaled_mm(mm, table: np.ndarray):
    one = _code_of(table, 1.0)
    # all-ones operands with distinct power-of-two per-channel scales
    M, N, K = 3, 14, 40
    qa = np.full((M, K), one, np.uint8)
    qw = np.full((N, K), one, np.uint8)
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    y = mm(qa, qw, np.float32(0.5), sw)
    assert y.shape == (M, N)
    want = np.array([[K * 0.5 * 2.0 ** (n % 7 - 3) for n in range(N)]] * M)
    assert np.array_equal(y, want), (y, want)
    # per-tensor weight scale
    y = mm(qa, qw, np.float32(0.25), np.array([3.0], np.float32))
    assert np.array_equal(y, np.full((M, N), K * 0.75))
    # permutation weights: y[m, n] = sa sw[n] dec(qa[m, pi(n)])
    K = N = 16
    pi = [(5 * n + 3) % K for n in range(N)]
    assert any(pi[pi[n]] != n for n in range(N))  # not an involution
    rng = np.random.default_rng(7)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(finite, size=(5, K)).astype(np.uint8)
    qw = np.zeros((N, K), np.uint8)
    for n in range(N):
        qw[n, pi[n]] = one
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    y = mm(qa, qw, np.float32(0.125), sw)
    want = np.array([[0.125 * sw[n] * table[qa[m, pi[n]]] for n in range(N)] for m in range(5)])
    assert np.array_equal(y, want)
    # exact integer arithmetic on codes in {-2,-1,-0.5,0,0.5,1,2}
    vals = [-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0]
    codes = np.array([_code_of(table, v) for v in vals], np.uint8)
    M, N, K = 7, 9, 33
    ia = rng.integers(0, len(vals), size=(M, K))
    iw = rng.integers(0, len(vals), size=(N, K))
    qa, qw = codes[ia], codes[iw]
    sa = np.float32(0.75)
    sw = np.array([2.0 ** -(n % 3) for n in range(N)], np.float32)
    y = mm(qa, qw, sa, sw)
    twice = [int(2 * v) for v in vals]
    for m in range(M):
        for n in range(N):
            acc4 = sum(twice[ia[m, k]] * twice[iw[n, k]] for k in range(K))
            assert y[m, n] == 0.75 * float(sw[n]) * acc4 / 4.0, (m, n)


def check_scaled_mm_per_token(mm, table: np.ndarray):
    """Pins of the product with one activation scale per row (per token):
    y[m, n] = sa[m] * sw(n) * sum_k dec(qa[m,k]) dec(qw[n,k])."""
    one = _code_of(table, 1.0)
    # all-ones operands, distinct power-of-two row and column scales, M != N
    # (a scale indexed by the column, or taken from one row, fails)
    M, N, K = 5, 12, 24
    qa = np.full((M, K), one, np.uint8)
    qw = np.full((N, K), one, np.uint8)
    sa = np.array([2.0 ** (m - 2) for m in range(M)], np.float32)
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    y = mm(qa, qw, sa, sw)
    assert y.shape == (M, N)
    want = np.array([[K * 2.0 ** (m - 2) * 2.0 ** (n % 7 - 3) for n in range(N)]
                     for m in range(M)])
    assert np.array_equal(y, want), (y, want)
    # per-tensor weight scale
    y = mm(qa, qw, sa, np.array([3.0], np.float32))
    assert np.array_equal(y, np.array([[K * 3.0 * 2.0 ** (m - 2)] * N for m in range(M)]))
    # permutation weights: y[m, n] = sa[m] sw[n] dec(qa[m, pi(n)])
    K = N = 16
    pi = [(5 * n + 3) % K for n in range(N)]
    rng = np.random.default_rng(11)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    M = 6
    qa = rng.choice(finite, size=(M, K)).astype(np.uint8)
    qw = np.zeros((N, K), np.uint8)
    for n in range(N):
        qw[n, pi[n]] = one
    sa = np.array([2.0 ** (-m) for m in range(M)], np.float32)
    sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
    y = mm(qa, qw, sa, sw)
    want = np.array([[float(sa[m]) * float(sw[n]) * table[qa[m, pi[n]]] for n in range(N)]
                     for m in range(M)])
    assert np.array_equal(y, want)
    # one scale for every row reduces to the per-tensor product
    qa = rng.choice(finite, size=(4, 16)).astype(np.uint8)
    qw = rng.choice(finite, size=(8, 16)).astype(np.uint8)
    sw = np.array([2.0 ** -(n % 3) for n in range(8)], np.float32)
    same = mm(qa, qw, np.full(4, 0.375, np.float32), sw)
    assert np.array_equal(same, mm(qa, qw, np.float32(0.375), sw))
    # exact integer arithmetic on codes in {-2,-1,-0.5,0,0.5,1,2}
    vals = [-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0]
    codes = np.array([_code_of(table, v) for v in vals], np.uint8)
    M, N, K = 7, 9, 33
    ia = rng.integers(0, len(vals), size=(M, K))
    iw = rng.integers(0, len(vals), size=(N, K))
    sa = np.array([0.75 * 2.0 ** -(m % 4) for m in range(M)], np.float32)
    sw = np.array([2.0 ** -(n % 3) for n in range(N)], np.float32)
    y = mm(codes[ia], codes[iw], sa, sw)
    twice = [int(2 * v) for v in vals]
    for m in range(M):
        for n in range(N):
            acc4 = sum(twice[ia[m, k]] * twice[iw[n, k]] for k in range(K))
            assert y[m, n] == float(sa[m]) * float(sw[n]) * acc4 / 4.0, (m, n)


# ---------------------------------------------------------------------------
# W8A16 product: ``fn(x_torch16, qw, sw) -> y float64 [M, N]``

def check_w8a16(fn, table: np.ndarray):
    one = _code_of(table, 1.0)
    M, N, K = 2, 10, 24
    x = torch.ones((M, K), dtype=torch.float16)
    qw = np.full((N, K), one, np.uint8)
    sw = np.array([2.0 ** (n % 7 - 3) for n in range(N)], np.float32)
    y = fn(x, qw, sw)
    assert y.shape == (M, N)
    assert np.array_equal(y, np.array([[K * s for s in sw]] * M, np.float64))
    # permutation weights: y[m, n] = sw[n] x[m, pi(n)]
    K = N = 16
    pi = [(5 * n + 3) % K for n in range(N)]
    g = torch.Generator().manual_seed(3)
    for dt in (torch.float16, torch.bfloat16):
        x = torch.randn((3, K), generator=g).to(dt)
        qw = np.zeros((N, K), np.uint8)
        for n in range(N):
            qw[n, pi[n]] = one
        sw = np.array([2.0 ** (n % 5 - 2) for n in range(N)], np.float32)
        y = fn(x, qw, sw)
        xf = x.double().numpy()
        want = np.array([[sw[n] * xf[m, pi[n]] for n in range(N)] for m in range(3)])
        assert np.array_equal(y, want)
    # exact integer arithmetic
    vals = [-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0]
    codes = np.array([_code_of(table, v) for v in vals], np.uint8)
    rng = np.random.default_rng(11)
    M, N, K = 4, 6, 48
    xi = rng.integers(-8, 9, size=(M, K))
    iw = rng.integers(0, len(vals), size=(N, K))
    x = torch.tensor(xi, dtype=torch.float16)
    qw = codes[iw]
    sw = np.array([2.0 ** -(n % 4) for n in range(N)], np.float32)
    y = fn(x, qw, sw)
    twice = [int(2 * v) for v in vals]
    for m in range(M):
        for n in range(N):
            acc2 = sum(int(xi[m, k]) * twice[iw[n, k]] for k in range(K))
            assert y[m, n] == float(sw[n]) * acc2 / 2.0, (m, n)


# ---------------------------------------------------------------------------
# Parity criteria.  The GPU parity tests of every floating-point product go
# through these acceptance functions, so they are pinned like the arithmetic:
# hand-built (y, y_ref) pairs just inside and just outside each bound.

def _ones_case(delta_one=0.0, delta_all=0.0, scale=1.0):
    """y_ref = scale * ones(10, 10) (rms = scale, ||y_ref||_F = 10 scale);
    y = y_ref with every element moved by delta_all * scale and element
    (3, 4) moved further by delta_one * scale."""
    y_ref = np.full((10, 10), scale, np.float64)
    y = y_ref + delta_all * scale
    y[3, 4] += delta_one * scale
    return y, y_ref


def check_gemm_close(close):
    """``close(y, y_ref) -> {"ok": bool, ...}``: elementwise
    |y - y_ref| <= 1e-2 (|y_ref| + rms(y_ref)) and relative Frobenius error
    <= 5e-3, the bound built from the reference alone."""
    for scale in (1.0, 1e3, 1e-3):
        # identical outputs pass
        y, r = _ones_case(scale=scale)
        assert close(y, r)["ok"]
        # one element at 0.95 of its bound (0.02 scale): the Frobenius error
        # is 0.0019, so the elementwise bound alone decides
        y, r = _ones_case(delta_one=0.019, scale=scale)
        assert close(y, r)["ok"], scale
        # ... and at 1.005 of it, upwards: a bound built from y (which has
        # grown) instead of y_ref would admit this one
        y, r = _ones_case(delta_one=0.0201, scale=scale)
        assert not close(y, r)["ok"], scale
        # every element moved by 0.00498 (elementwise ratio 0.25): Frobenius
        # 0.00498 passes, 0.00502 fails; dividing by ||y|| instead of
        # ||y_ref|| would pass the latter (0.004995)
        y, r = _ones_case(delta_all=0.00498, scale=scale)
        assert close(y, r)["ok"], scale
        y, r = _ones_case(delta_all=0.00502, scale=scale)
        assert not close(y, r)["ok"], scale
        # the same error downwards
        y, r = _ones_case(delta_all=-0.00502, scale=scale)
        assert not close(y, r)["ok"], scale
    # the elementwise bound has the rms term: an element whose reference is
    # zero may be off by up to 1e-2 rms(y_ref)
    y, r = _ones_case()
    r[0, 0] = 0.0
    rms = float(np.sqrt(np.mean(r ** 2)))
    y[0, 0] = 0.0098 * rms
    assert close(y, r)["ok"]
    y[0, 0] = 0.0102 * rms
    assert not close(y, r)["ok"]
    # an all-zero reference admits only an all-zero output
    z = np.zeros((4, 6))
    assert close(z.copy(), z)["ok"]
    y = z.copy()
    y[2, 3] = 1e-30
    assert not close(y, z)["ok"]
    # non-finite outputs are rejected
    for bad in (np.nan, np.inf, -np.inf):
        y, r = _ones_case()
        y[1, 1] = bad
        assert not close(y, r)["ok"], bad
    # empty outputs pass
    assert close(np.zeros((0, 5)), np.zeros((0, 5)))["ok"]


def brute_midpoint_distance(t, table: np.ndarray) -> np.ndarray:
    """Independent restatement: the distance from min(|t|, 448) to the
    nearest of the 126 midpoints between consecutive non-negative finite
    E4M3 values, by a scan over all of them."""
    pos = table[:127]
    mids = [(pos[i] + pos[i + 1]) / 2 for i in range(126)]
    out = []
    for v in np.asarray(t, np.float64).reshape(-1):
        a = min(abs(v), 448.0)
        out.append(min(abs(a - m) for m in mids))
    return np.array(out)


def check_midpoint_distance(dist, table: np.ndarray):
    """``dist(t) -> distance of each |t| (clipped to 448) to the nearest
    rounding midpoint of E4M3``."""
    # hand values: a midpoint itself; a code value (1.0 sits between the
    # midpoints 0.96875 and 1.0625); zero (first midpoint 2^-10); beyond the
    # largest value (clipped to 448, the last midpoint is 432); the sign
    t = np.array([1.0625, 1.0, -1.0, 0.0, 2.0 ** -10, 500.0, 448.0, -3.0 * 2.0 ** -10])
    want = np.array([0.0, 0.03125, 0.03125, 2.0 ** -10, 0.0, 16.0, 16.0, 0.0])
    got = np.asarray(dist(t), np.float64)
    assert np.array_equal(got, want), (got, want)
    # against the scan on every code value, every midpoint, and points in
    # between, both signs
    pos = table[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(5)
    t = np.concatenate([pos, mids, mids * (1 + 1e-3), mids * (1 - 1e-3),
                        rng.uniform(0, 460, 500), np.exp2(rng.uniform(-12, 9, 500))])
    t = np.concatenate([t, -t])
    got = np.asarray(dist(t), np.float64)
    want = brute_midpoint_distance(t, table)
    assert np.array_equal(got, want)


def check_e4m3_output_close(close, table: np.ndarray):
    """``close(codes, y_ref, out_scale) -> {"ok": bool, ...}`` for E4M3
    product outputs: codes within one step of c_ref = E4M3(y_ref / os)
    (0x00 and 0x80 equal), equal to c_ref wherever t = y_ref / os is
    farther than 1e-3 (|t| + rms(t)) from a rounding midpoint, and
    ||dec(code) - clip(t)||_F <= 2^-4 ||clip(t)||_F."""
    enc = {float(table[c]): c for c in range(127)}
    os_ = np.float32(0.5)
    # t = 1.0 for every element (the code 0x38); far from both midpoints
    # (0.03125 away; the window is 2e-3)
    t = np.full((4, 8), 1.0)
    y_ref = t * np.float64(os_)
    c = np.full(t.shape, enc[1.0], np.uint8)
    assert close(c, y_ref, os_)["ok"]
    # one step off there is rejected (a window grown 1000-fold would let it
    # through), and so is every other wrong code far from a midpoint
    for wrong in (enc[1.125], enc[0.9375]):
        cc = c.copy()
        cc[1, 2] = wrong
        assert not close(cc, y_ref, os_)["ok"], hex(wrong)
    # t just below the midpoint 1.0625 (inside the window): c_ref = 0x38
    # (1.0); the neighbour 0x39 (1.125) is accepted, 0x3A (1.25) is not
    t = np.full((4, 8), 1.0)
    t[2, 5] = 1.0625 - 1e-4
    y_ref = t * np.float64(os_)
    cc = np.full(t.shape, enc[1.0], np.uint8)
    assert close(cc, y_ref, os_)["ok"]
    cc[2, 5] = enc[1.125]
    assert close(cc, y_ref, os_)["ok"]
    cc[2, 5] = enc[1.25]
    assert not close(cc, y_ref, os_)["ok"]
    # a wrong sign is many steps away
    cc[2, 5] = 0x80 | enc[1.0]
    assert not close(cc, y_ref, os_)["ok"]
    # signed zero: tiny negative references round to 0x80; 0x00 is the same
    # value and is accepted, in both directions.  (Beside 16 values of 0.5,
    # which keep the Frobenius error small and the window at ~5e-4.)
    half = np.full(16, enc[0.5], np.uint8)
    t = np.concatenate([np.full(16, 0.5), [-1e-5, 1e-5, -1e-6]]).reshape(1, -1)
    y_ref = t * np.float64(os_)
    zeros = lambda a, b, c: np.concatenate([half, np.array([a, b, c], np.uint8)]).reshape(1, -1)
    assert close(zeros(0x80, 0x00, 0x80), y_ref, os_)["ok"]
    assert close(zeros(0x00, 0x80, 0x00), y_ref, os_)["ok"]
    # ... but the smallest subnormal is a step away from zero and t = -1e-5
    # is far from the first midpoint (2^-10): rejected
    assert not close(zeros(0x81, 0x00, 0x80), y_ref, os_)["ok"]
    # saturated references: |t| >= 448 must give 0x7E / 0xFE; 0x7D (416) is
    # a step below, far from any midpoint of the clipped value
    t = np.array([[1000.0, -600.0, 448.0, 1.0]])
    y_ref = t * np.float64(os_)
    good = np.array([[0x7E, 0xFE, 0x7E, enc[1.0]]], np.uint8)
    res = close(good, y_ref, os_)
    assert res["ok"] and res["rel_fro"] == 0.0, res
    bad = good.copy()
    bad[0, 0] = 0x7D
    assert not close(bad, y_ref, os_)["ok"]
    # the Frobenius bound: references on the midpoint between the two
    # smallest subnormals (1.5 * 2^-9) carry a relative error of 1/3 even
    # with the nearest codes, which the bound rejects
    t = np.full((2, 3), 1.5 * 2.0 ** -9)
    y_ref = t * np.float64(os_)
    res = close(np.full(t.shape, 0x02, np.uint8), y_ref, os_)
    assert not res["ok"] and res["max_step"] == 0, res
    # NaN codes are rejected
    t = np.full((2, 2), 1.0)
    cc = np.full(t.shape, enc[1.0], np.uint8)
    cc[0, 1] = 0x7F
    assert not close(cc, t * np.float64(os_), os_)["ok"]
    # the output scale divides: the same codes against y_ref = 4 os t pass
    # only with the codes of 4 t
    t = np.full((3, 3), 1.0)
    y_ref = 4.0 * t * np.float64(os_)
    assert close(np.full(t.shape, enc[4.0], np.uint8), y_ref, os_)["ok"]
    assert not close(np.full(t.shape, enc[1.0], np.uint8), y_ref, os_)["ok"]


# ---------------------------------------------------------------------------
# RMS normalization: ``norm(x_torch16 [M, K], gamma_torch16 [K], eps) ->
# h float64 [M, K]`` (h = x gamma / sqrt(mean_k x^2 + eps) per row)

def check_rmsnorm(norm):
    # constant rows, eps = 0: every h is +-gamma exactly (c^2 and sqrt(c^2)
    # are exact); rows of different constants are independent
    K = 48
    g = torch.Generator().manual_seed(1)
    gamma = (torch.rand(K, generator=g) + 0.5).to(torch.bfloat16)
    x = torch.tensor([[1.5] * K, [-0.375] * K, [96.0] * K], dtype=torch.bfloat16)
    h = norm(x, gamma, 0.0)
    gf = gamma.double().numpy()
    want = np.stack([gf, -gf, gf])
    assert np.array_equal(h, want), (h - want)
    # eps = 3 c^2: the root is 2|c|, h = +-gamma / 2 exactly
    h = norm(x[:1], gamma, 3 * 1.5 ** 2)
    assert np.array_equal(h, gf[None, :] / 2)
    # a single nonzero element a in a row of K = 64: mean = a^2 / 64, the
    # root is |a| / 8, so h = 8 sign(a) gamma there and 0 elsewhere
    K = 64
    gamma = torch.linspace(0.5, 2.0, K).to(torch.bfloat16)
    x = torch.zeros((2, K), dtype=torch.bfloat16)
    x[0, 5] = 3.0
    x[1, 60] = -0.25
    h = norm(x, gamma, 0.0)
    gf = gamma.double().numpy()
    want = np.zeros((2, K))
    want[0, 5] = 8 * gf[5]
    want[1, 60] = -8 * gf[60]
    assert np.array_equal(h, want)
    # random rows, gamma = 1, eps = 0: mean(h^2) = 1 per row; powers of two
    # of x leave h unchanged; permuting the columns of x and gamma together
    # permutes h
    x = torch.randn((5, 96), generator=g).to(torch.bfloat16)
    ones = torch.ones(96, dtype=torch.bfloat16)
    h = norm(x, ones, 0.0)
    assert np.allclose((h ** 2).mean(axis=1), 1.0, rtol=1e-13)
    assert np.array_equal(norm((x.float() * 8).to(torch.bfloat16), ones, 0.0), h)
    gamma = (torch.rand(96, generator=g) + 0.5).to(torch.bfloat16)
    perm = torch.randperm(96, generator=g)
    h = norm(x, gamma, 1e-5)
    hp = norm(x[:, perm], gamma[perm], 1e-5)
    assert np.array_equal(hp, h[:, perm.numpy()])
    # eps matters: against the closed form sqrt(ms / (ms + eps)) of mean(h^2)
    h = norm(x, ones, 0.5)
    ms = (x.double().numpy() ** 2).mean(axis=1)
    assert np.allclose((h ** 2).mean(axis=1), ms / (ms + 0.5), rtol=1e-13)


# ``rnd(v float64 array, dtype) -> float64 array`` of the nearest bf16 /
# fp16 values, ties to even
def check_round_to(rnd):
    for dt in (torch.bfloat16, torch.float16):
        one = 1.0
        p = 8 if dt == torch.bfloat16 else 11
        u = 2.0 ** -(p - 1)  # spacing at 1
        # ties: 1 + u/2 -> 1 (even), 1 + 3u/2 -> 1 + 2u (even)
        got = rnd(np.array([one + u / 2, one + 3 * u / 2, -(one + u / 2), one + u / 2 + 2.0 ** -40]), dt)
        assert np.array_equal(got, [1.0, 1.0 + 2 * u, -1.0, 1.0 + u]), (dt, got)
        # the library cast of float32 values (one rounding) agrees, including
        # subnormals of the format and values right at midpoints
        rng = np.random.default_rng(3)
        v = (rng.standard_normal(100_000) * np.exp2(rng.uniform(-30, 14, 100_000))).astype(np.float32)
        lib = torch.from_numpy(v).to(dt).double().numpy()
        assert np.array_equal(rnd(v.astype(np.float64), dt), lib), dt
        vals = torch.from_numpy(all_16bit_values(dt)).double().numpy()
        vals = np.unique(vals[np.isfinite(vals) & (vals > 0)])
        mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact in float32
        lib = torch.from_numpy(mids).to(dt).double().numpy()
        assert np.array_equal(rnd(mids.astype(np.float64), dt), lib), dt


# ``close(h, h_ref, dtype) -> {"ok": ...}``: h must be the rounding of h_ref,
# or either neighbour within a relative window 2^-16 of a midpoint
def check_rounded_close(close):
    dt = torch.bfloat16
    u = 2.0 ** -7
    h_ref = np.array([1.0 + 0.3 * u, 2.0 + 2 * 0.7 * u, -3.0])
    want = np.array([1.0, 2.0 + 2 * u, -3.0])
    assert close(want, h_ref, dt)["ok"]
    # one unit off far from a midpoint: rejected, in either direction
    for i, d in ((0, u), (1, -2 * u), (2, 2 * u)):
        h = want.copy()
        h[i] += d
        assert not close(h, h_ref, dt)["ok"], (i, d)
    # h_ref just above the midpoint 1 + u/2 (inside the window): 1 + u is the
    # rounding, 1 is accepted too, 1 + 2u is not
    h_ref = np.array([1.0 + u / 2 + 2.0 ** -22])
    assert close(np.array([1.0 + u]), h_ref, dt)["ok"]
    assert close(np.array([1.0]), h_ref, dt)["ok"]
    assert not close(np.array([1.0 + 2 * u]), h_ref, dt)["ok"]
    # ... but 2^-14 above it is outside the window: only 1 + u
    h_ref = np.array([1.0 + u / 2 + 2.0 ** -14])
    assert close(np.array([1.0 + u]), h_ref, dt)["ok"]
    assert not close(np.array([1.0]), h_ref, dt)["ok"]
    # non-finite results are rejected
    assert not close(np.array([np.nan]), np.array([1.0]), dt)["ok"]
    assert not close(np.array([np.inf]), np.array([1.0]), dt)["ok"]


# ---------------------------------------------------------------------------
# Grouped W8A8 product (mixture of experts):
# ``gmm(qa [M, K], qw [E, N, K], offsets [E+1], sa (1 or M), sw (E or E x N))
# -> y float64 [M, N]``; rows outside every group are 0

def check_grouped_mm(gmm, table: np.ndarray):
    one = _code_of(table, 1.0)
    # all-ones operands: y[m, n] = K sa sw_e(n) for m in group e; groups of
    # different sizes, an empty group, rows after the last group
    E, N, K, M = 4, 32, 48, 23
    offs = np.array([0, 5, 5, 16, 20], np.int32)  # expert 1 empty; rows 20..22 unrouted
    qa = np.full((M, K), one, np.uint8)
    qw = np.full((E, N, K), one, np.uint8)
    sw = np.array([[2.0 ** (e - 2) * 2.0 ** (n % 5 - 2) for n in range(N)] for e in range(E)],
                  np.float32)
    y = gmm(qa, qw, offs, np.float32(0.5), sw)
    assert y.shape == (M, N)
    want = np.zeros((M, N))
    for e in range(E):
        want[offs[e]:offs[e + 1]] = K * 0.5 * sw[e][None, :]
    assert np.array_equal(y, want), np.argwhere(y != want)[:5]
    # one scale per expert
    sw1 = np.array([[3.0], [5.0], [0.25], [7.0]], np.float32)
    y = gmm(qa, qw, offs, np.float32(0.5), sw1)
    want = np.zeros((M, N))
    for e in range(E):
        want[offs[e]:offs[e + 1]] = K * 0.5 * sw1[e, 0]
    assert np.array_equal(y, want)
    # a different permutation per expert: y[m, n] = sa sw_e[n] dec(qa[m, pi_e(n)])
    K = N = 16
    E, M = 3, 12
    offs = np.array([0, 4, 9, 12], np.int32)
    rng = np.random.default_rng(13)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(finite, size=(M, K)).astype(np.uint8)
    pis = [[(a * n + b) % K for n in range(N)] for a, b in ((5, 3), (7, 1), (3, 10))]
    qw = np.zeros((E, N, K), np.uint8)
    for e in range(E):
        for n in range(N):
            qw[e, n, pis[e][n]] = one
    sw = np.array([[2.0 ** ((n + e) % 5 - 2) for n in range(N)] for e in range(E)], np.float32)
    sa = np.array([2.0 ** -(m % 3) for m in range(M)], np.float32)  # per token
    y = gmm(qa, qw, offs, sa, sw)
    want = np.zeros((M, N))
    for e in range(E):
        for m in range(offs[e], offs[e + 1]):
            for n in range(N):
                want[m, n] = float(sa[m]) * float(sw[e, n]) * table[qa[m, pis[e][n]]]
    assert np.array_equal(y, want)
    # exact integer arithmetic against Python integers
    vals = [-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0]
    codes = np.array([_code_of(table, v) for v in vals], np.uint8)
    E, M, N, K = 3, 10, 5, 40
    offs = np.array([0, 2, 7, 10], np.int32)
    ia = rng.integers(0, len(vals), size=(M, K))
    iw = rng.integers(0, len(vals), size=(E, N, K))
    sw = np.array([[0.5], [2.0], [0.125]], np.float32)
    y = gmm(codes[ia], codes[iw], offs, np.float32(0.75), sw)
    twice = [int(2 * v) for v in vals]
    for e in range(E):
        for m in range(offs[e], offs[e + 1]):
            for n in range(N):
                acc4 = sum(twice[ia[m, k]] * twice[iw[e, n, k]] for k in range(K))
                assert y[m, n] == 0.75 * float(sw[e, 0]) * acc4 / 4.0, (e, m, n)
