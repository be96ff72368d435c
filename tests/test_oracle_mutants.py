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


# ---------------------------------------------------------------------------
# parity criteria: copies of the acceptance functions with planted mistakes

def _gemm_close_mutant(mistake):
    def close(y, y_ref):
        y = np.asarray(y, np.float64)
        y_ref = np.asarray(y_ref, np.float64)
        if y.size == 0:
            return {"ok": True}
        ref_for_bound = y if mistake == "bound_from_y" else y_ref
        rms = float(np.sqrt(np.mean(ref_for_bound ** 2)))
        err = np.abs(y - y_ref)
        term = 0.0 if mistake == "no_rms_term" else rms
        bound = 1e-2 * (np.abs(ref_for_bound) + term)
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
        max_ratio = float(np.max(ratio))
        denom = {"fro_over_y_norm": np.linalg.norm(y), "abs_fro": 1.0}.get(
            mistake, np.linalg.norm(y_ref))
        num = np.linalg.norm(y - y_ref)
        if mistake == "squared_fro":
            num, denom = num ** 2, denom ** 2
        rel = float(num / denom) if denom > 0 else float(np.linalg.norm(y))
        finite = bool(np.all(np.isfinite(y)))
        fro_ok = True if mistake == "elementwise_only" else rel <= 5e-3
        return {"ok": finite and max_ratio <= 1.0 and fro_ok}
    return close


@pytest.mark.parametrize("mistake", ["bound_from_y", "no_rms_term", "fro_over_y_norm",
                                     "abs_fro", "squared_fro", "elementwise_only"])
def test_gemm_close_mutants_rejected(mistake):
    with pytest.raises(AssertionError):
        pins.check_gemm_close(_gemm_close_mutant(mistake))


def test_gemm_close_copy_without_mistake_passes():
    pins.check_gemm_close(_gemm_close_mutant(None))


def _midpoint_mutant(mistake, table):
    def dist(t):
        pos = table[:127]
        mids = (pos[:-1] + pos[1:]) / 2
        a = np.asarray(t, np.float64)
        a = a if mistake == "no_abs" else np.abs(a)
        if mistake != "no_clip":
            a = np.minimum(a, 448.0)
        i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
        if mistake == "off_by_one":
            i = np.clip(i + 1, 1, len(mids) - 1)
        if mistake == "one_side":
            return np.abs(a - mids[i])
        return np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))
    return dist


@pytest.mark.parametrize("mistake", ["no_abs", "no_clip", "off_by_one", "one_side"])
def test_midpoint_mutants_rejected(table, mistake):
    with pytest.raises(AssertionError):
        pins.check_midpoint_distance(_midpoint_mutant(mistake, table), table)


def test_midpoint_copy_without_mistake_passes(table):
    pins.check_midpoint_distance(_midpoint_mutant(None, table), table)


def _e4m3_close_mutant(mistake, table):
    def ordinal(c):
        c = np.asarray(c, np.int64)
        mag = c & 0x7F
        if mistake == "signed_zero_distinct":
            return np.where(c & 0x80, -mag - 1, mag)
        return np.where(c & 0x80, -mag, mag)

    def close(codes, y_ref, out_scale):
        codes = np.asarray(codes, np.uint8)
        y_ref = np.asarray(y_ref, np.float64)
        os_ = np.float64(np.float32(out_scale))
        t = y_ref if mistake == "scale_not_divided" else y_ref / os_
        c_ref = oracle.e4m3_encode(t)
        step = np.abs(ordinal(codes) - ordinal(c_ref))
        rms = float(np.sqrt(np.mean(t ** 2)))
        window = 1e-3 * (1000.0 if mistake == "window_x1000" else 1.0)
        far = oracle._nearest_midpoint_distance(t) > window * (np.abs(t) + rms)
        exact_bad = int(np.count_nonzero(far & (step != 0)))
        if mistake == "no_exactness":
            exact_bad = 0
        tc = np.clip(t, -448.0, 448.0)
        dec = table[codes]
        nref = float(np.linalg.norm(tc))
        rel = float(np.linalg.norm(dec - tc) / nref) if nref > 0 else float(np.linalg.norm(dec))
        max_step = int(step.max()) if step.size else 0
        allowed = 2 if mistake == "two_steps" else 1
        fro_ok = True if mistake == "no_fro" else rel <= 2.0 ** -4
        ok = max_step <= allowed and exact_bad == 0 and fro_ok and not np.any(np.isnan(dec))
        return {"ok": ok, "max_step": max_step, "rel_fro": rel}
    return close


@pytest.mark.parametrize("mistake", ["signed_zero_distinct", "scale_not_divided",
                                     "window_x1000", "no_exactness", "two_steps", "no_fro"])
def test_e4m3_close_mutants_rejected(table, mistake):
    with pytest.raises(AssertionError):
        pins.check_e4m3_output_close(_e4m3_close_mutant(mistake, table), table)


def test_e4m3_close_copy_without_mistake_passes(table):
    pins.check_e4m3_output_close(_e4m3_close_mutant(None, table), table)


# ---------------------------------------------------------------------------
# RMS normalization, 16-bit rounding and its acceptance function

def _norm_mutant(mistake):
    def norm(x, gamma, eps):
        X = oracle.widen(x).astype(np.float64)
        G = oracle.widen(gamma).astype(np.float64).reshape(-1)
        axis = 0 if mistake == "over_columns" else 1
        ss = (X ** 2).sum(axis=axis, keepdims=True)
        ms = ss if mistake == "sum_not_mean" else ss / X.shape[axis]
        if mistake == "eps_outside_sqrt":
            rms = np.sqrt(ms) + eps
        elif mistake == "no_sqrt":
            rms = ms + eps
        else:
            rms = np.sqrt(ms + eps)
        if mistake == "gamma_reversed":
            G = G[::-1]
        if mistake == "gamma_divides":
            return X / G / rms
        return X * G / rms
    return norm


@pytest.mark.parametrize("mistake", ["over_columns", "sum_not_mean", "eps_outside_sqrt",
                                     "no_sqrt", "gamma_reversed", "gamma_divides"])
def test_rmsnorm_mutants_rejected(mistake):
    with pytest.raises(AssertionError):
        pins.check_rmsnorm(_norm_mutant(mistake))


def test_rmsnorm_copy_without_mistake_passes():
    pins.check_rmsnorm(_norm_mutant(None))


def _round_mutant(mistake):
    def rnd(v, dtype):
        p, emin = oracle.FORMATS[oracle._fmt(dtype)]
        v = np.asarray(v, np.float64)
        out = np.empty_like(v)
        for i, x in enumerate(v.reshape(-1)):
            if x == 0:
                out.reshape(-1)[i] = x
                continue
            e = max(int(np.floor(np.log2(abs(x)))), emin)
            if mistake == "flush_subnormals" and abs(x) < 2.0 ** emin:
                out.reshape(-1)[i] = 0.0
                continue
            ulp = 2.0 ** (e - (p - 1))
            t = x / ulp
            if mistake == "ties_away":
                r = np.sign(t) * np.floor(abs(t) + 0.5)
            elif mistake == "truncate":
                r = np.trunc(t)
            else:
                r = np.rint(t)
            out.reshape(-1)[i] = r * ulp
        return out
    return rnd


@pytest.mark.parametrize("mistake", ["ties_away", "truncate", "flush_subnormals"])
def test_round_to_mutants_rejected(mistake):
    with pytest.raises(AssertionError):
        pins.check_round_to(_round_mutant(mistake))


def _rounded_close_mutant(mistake):
    def close(h, h_ref, dtype):
        h = np.asarray(h, np.float64)
        h_ref = np.asarray(h_ref, np.float64)
        window = {"window_x1000": 2.0 ** -16 * 1000, "no_window": 0.0}.get(mistake, 2.0 ** -16)
        want = oracle.round_to(h_ref, dtype)
        lo = oracle.round_to(h_ref * (1 - window), dtype)
        hi = oracle.round_to(h_ref * (1 + window), dtype)
        ok = (h == want) | (h == lo) | (h == hi)
        if mistake == "nan_ok":
            ok |= np.isnan(h)
        return {"ok": bool(np.all(ok))}
    return close


@pytest.mark.parametrize("mistake", ["window_x1000", "no_window", "nan_ok"])
def test_rounded_close_mutants_rejected(mistake):
    with pytest.raises(AssertionError):
        pins.check_rounded_close(_rounded_close_mutant(mistake))


def test_rounded_close_copy_without_mistake_passes():
    pins.check_rounded_close(_rounded_close_mutant(None))


# ---------------------------------------------------------------------------
# grouped product

def _grouped_mutant(mistake, table):
    def gmm(qa, qw, offs, sa, sw):
        A = table[np.asarray(qa)]
        W = table[np.asarray(qw)]
        E, N, _ = W.shape
        M = A.shape[0]
        sw = np.asarray(sw, np.float64).reshape(E, -1)
        sa = np.asarray(sa, np.float64).reshape(-1)
        y = np.zeros((M, N))
        for e in range(E):
            lo, hi = int(offs[e]), int(offs[e + 1])
            if mistake == "inclusive_end":
                hi = min(hi + 1, M)
            ew = (e + 1) % E if mistake == "next_expert" else e
            es = 0 if mistake == "first_expert_scale" else e
            for m in range(lo, hi):
                scol = sw[es] if sw.shape[1] == N else np.full(N, sw[es, 0])
                if mistake == "flat_channel_scale" and sw.shape[1] == N:
                    scol = sw.reshape(-1)[:N]
                s_m = sa[m] if sa.size == M and M != 1 else sa[0]
                y[m] = (A[m] @ W[ew].T) * s_m * scol
        return y
    return gmm


@pytest.mark.parametrize("mistake", ["inclusive_end", "next_expert", "first_expert_scale",
                                     "flat_channel_scale"])
def test_grouped_mutants_rejected(table, mistake):
    with pytest.raises(AssertionError):
        pins.check_grouped_mm(_grouped_mutant(mistake, table), table)


def test_grouped_copy_without_mistake_passes(table):
    pins.check_grouped_mm(_grouped_mutant(None, table), table)
