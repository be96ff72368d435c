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
