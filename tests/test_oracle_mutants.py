"""Plant plausible mistakes in copies of the oracle's arithmetic (on the CPU)
and check that the pins reject every one of them.  This shows that the pins
of test_oracle_*.py can tell a wrong oracle from a right one."""
import numpy as np
import pytest
import torch

import oracle
import pins


@pytest.fixture(scope="module")
def table():
    return oracle.decode_table()


def _nearest(values, table, tie):
    """Copy of the oracle's nearest-code encode with a pluggable tie rule and
    switches for the planted mistakes."""
    pos = table[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    out = np.empty(len(values), np.uint8)
    for i, v in enumerate(np.asarray(values, np.float64)):
        if np.isnan(v):
            out[i] = 0x7F
            continue
        sign = 0x80 if np.signbit(v) else 0
        a = abs(v)
        if a >= 448.0 and tie != "nosat":
            out[i] = sign | 0x7E
            continue
        if a >= 464.0:  # no saturation: overflow becomes NaN
            out[i] = 0x7F
            continue
        lo = int(np.searchsorted(pos, a, side="right") - 1)
        lo = min(lo, 125)
        hi = lo + 1
        if a < mids[lo]:
            c = lo
        elif a > mids[lo]:
            c = hi
        elif tie == "away":
            c = hi
        elif tie == "trunc":
            c = lo
        else:
            c = lo if lo % 2 == 0 else hi
        if tie == "trunc":
            c = lo
        if tie == "unsigned_zero" and c == 0:
            sign = 0
        out[i] = sign | c
    return out


@pytest.mark.parametrize("mistake", ["away", "trunc", "nosat", "unsigned_zero"])
def test_encoder_mutants_rejected(table, mistake):
    with pytest.raises(AssertionError):
        pins.check_encoder(lambda v: _nearest(v, table, mistake), table)


def test_encoder_copy_without_mistake_passes(table):
    # the harness itself is sound: the unmutated copy passes the golden part
    vals = np.array([v for v, _ in pins.load_rounding()])
    want = np.array([c for _, c in pins.load_rounding()], np.uint8)
    assert np.array_equal(_nearest(vals, table, "even"), want)


def _quant_mutant(mistake):
    def quant(x, scale=None):
        xf = oracle.widen(x).reshape(-1)
        if scale is None:
            if mistake == "no_abs":
                amax = np.float32(xf.max())
            else:
                amax = np.float32(np.abs(xf).max())
            const = np.float32(240.0) if mistake == "const240" else np.float32(448.0)
            s = np.float32(amax / const)
            if mistake == "bf16_scale":
                s = np.float32(torch.tensor(float(s)).to(torch.bfloat16).item())
            if s == 0:
                s = np.float32(1.0)
        else:
            s = np.float32(scale)
        q = oracle.e4m3_encode((xf / s).astype(np.float32))
        return q, s
    return quant


@pytest.mark.parametrize("mistake", ["no_abs", "const240", "bf16_scale"])
def test_quant_mutants_rejected(table, mistake):
    quant = _quant_mutant(mistake)
    rejected = False
    try:
        pins.check_quant_worked(quant)
        for seed in range(3):
            g = torch.Generator().manual_seed(seed)
            x = torch.randn(500, generator=g).to(torch.bfloat16)
            pins.check_quant_invariants(quant, table, x)
    except AssertionError:
        rejected = True
    assert rejected


def test_quant_copy_without_mistake_passes(table):
    quant = _quant_mutant(None)
    pins.check_quant_worked(quant)
    pins.check_quant_invariants(quant, table, torch.randn(300).to(torch.bfloat16))


def _mm_mutant(mistake, table):
    def mm(qa, qw, sa, sw):
        A = table[np.asarray(qa)]
        W = table[np.asarray(qw)]
        N, K = W.shape
        sw = np.asarray(sw, np.float64).reshape(-1)
        if mistake == "transposed":
            acc = A @ W.reshape(K, N)
        elif mistake == "dropped_term":
            acc = A[:, 1:] @ W[:, 1:].T
        else:
            acc = A @ W.T
        if sw.size == 1:
            scale = np.full(N, sw[0])
        else:
            scale = sw[::-1] if mistake == "reversed_scales" else sw
        sa = np.float64(sa)
        if mistake == "no_act_scale":
            sa = 1.0
        return acc * (sa * scale).reshape(1, -1)
    return mm


@pytest.mark.parametrize("mistake", ["transposed", "dropped_term", "reversed_scales", "no_act_scale"])
def test_scaled_mm_mutants_rejected(table, mistake):
    with pytest.raises(AssertionError):
        pins.check_scaled_mm(_mm_mutant(mistake, table), table)


def test_scaled_mm_copy_without_mistake_passes(table):
    pins.check_scaled_mm(_mm_mutant(None, table), table)


def _per_token_mutant(mistake, table):
    def mm(qa, qw, sa, sw):
        A = table[np.asarray(qa)]
        W = table[np.asarray(qw)]
        M, N = A.shape[0], W.shape[0]
        sw = np.asarray(sw, np.float64).reshape(-1)
        scale_n = np.full(N, sw[0]) if sw.size == 1 else sw
        sa = np.asarray(sa, np.float64).reshape(-1)
        rows = np.full(M, sa[0]) if sa.size == 1 else sa
        scale = rows.reshape(-1, 1) * scale_n.reshape(1, -1)
        if mistake == "scale_by_column":
            # the row scale read at the column index: sa[n mod M]
            scale = np.array([[rows[n % M] * scale_n[n] for n in range(N)] for _ in range(M)])
        elif mistake == "first_row_scale":
            scale = rows[0] * np.tile(scale_n, (M, 1))
        elif mistake == "no_act_scale":
            scale = np.tile(scale_n, (M, 1))
        return (A @ W.T) * scale
    return mm


@pytest.mark.parametrize("mistake", ["scale_by_column", "first_row_scale", "no_act_scale"])
def test_per_token_mutants_rejected(table, mistake):
    with pytest.raises(AssertionError):
        pins.check_scaled_mm_per_token(_per_token_mutant(mistake, table), table)


def test_per_token_copy_without_mistake_passes(table):
    pins.check_scaled_mm_per_token(_per_token_mutant(None, table), table)


def _w8a16_mutant(mistake, table):
    def fn(x, qw, sw):
        X = oracle.widen(x).astype(np.float64)
        W = table[np.asarray(qw)]
        N, K = W.shape
        sw = np.asarray(sw, np.float64).reshape(-1)
        if mistake == "transposed":
            acc = X @ W.reshape(K, N)
        else:
            acc = X @ W.T
        if mistake == "no_scale":
            sw = np.ones_like(sw)
        if mistake == "x_rounded_to_e4m3":
            acc = table[oracle.e4m3_encode(X)] @ W.T
        return acc * sw.reshape(1, -1)
    return fn


@pytest.mark.parametrize("mistake", ["transposed", "no_scale", "x_rounded_to_e4m3"])
def test_w8a16_mutants_rejected(table, mistake):
    with pytest.raises(AssertionError):
        pins.check_w8a16(_w8a16_mutant(mistake, table), table)


def test_w8a16_copy_without_mistake_passes(table):
    pins.check_w8a16(_w8a16_mutant(None, table), table)
