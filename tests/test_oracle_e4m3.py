"""Pins of the oracle's OCP E4M3 decode and saturating round-to-nearest-even
encode ("RFC: FP8 Quantization Schema in vLLM", Scope: FP8_E4M3 (OCP))."""
import math

import numpy as np
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def table():
    return oracle.decode_table()


def test_decode_table(table):
    pins.check_decode_table(table)
    assert table[0x7E] == 448.0 and table[0x01] == 2.0 ** -9 and table[0x08] == 2.0 ** -6


def test_encode_pins(table):
    pins.check_encoder(oracle.e4m3_encode, table)


def test_encode_float32_entry_matches_float64_entry():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(50_000) * 100).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(v), oracle.e4m3_encode(v.astype(np.float64)))


def test_encode_against_linear_scan(table):
    # brute force on a few thousand values, including every midpoint and its
    # float32 neighbours
    vals = []
    pos = table[:127]
    for a, b in zip(pos[:-1], pos[1:]):
        mid = np.float32((a + b) / 2)
        vals += [float(mid), float(np.nextafter(mid, np.float32(0))),
                 float(np.nextafter(mid, np.float32(1000)))]
    rng = np.random.default_rng(9)
    vals += list((rng.standard_normal(3000) * np.exp2(rng.uniform(-12, 9, 3000))).astype(np.float32))
    vals = np.array(vals, np.float64)
    vals = np.concatenate([vals, -vals])
    got = oracle.e4m3_encode(vals)
    for v, c in zip(vals, got):
        assert c == pins.linear_scan_encode(float(v), table), (v, hex(c))


def test_encode_nan():
    assert oracle.e4m3_encode(np.array([math.nan]))[0] == 0x7F


def test_ml_dtypes_agrees(table):
    ml_dtypes = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    lib = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(table))
    assert np.array_equal(lib[~nan], table[~nan])
    v = pins.all_16bit_values(__import__("torch").float16)
    want = np.clip(v, -448, 448).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(v), want)
