"""Pins of the oracle's grouped product for mixture-of-experts layers ("RFC:
FP8 Quantization Schema in vLLM", the gate_proj question: FP8 products need
shapes divisible by 16; the experts' products are FP8, an 8-expert gate is
padded to 16 output channels here)."""
import numpy as np
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def table():
    return oracle.decode_table()


def test_grouped_bruteforce(table):
    pins.check_grouped_mm(oracle.grouped_mm_bruteforce, table)


def test_grouped_matmul_path(table):
    pins.check_grouped_mm(oracle.grouped_mm_ref, table)


def test_one_group_is_the_plain_product():
    rng = np.random.default_rng(4)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(finite, size=(9, 64)).astype(np.uint8)
    qw = rng.choice(finite, size=(1, 32, 64)).astype(np.uint8)
    sw = np.array([2.0 ** -(n % 4) for n in range(32)], np.float32)
    y = oracle.grouped_mm_bruteforce(qa, qw, np.array([0, 9], np.int32), np.float32(0.3), sw)
    assert np.array_equal(y, oracle.scaled_mm_bruteforce(qa, qw[0], np.float32(0.3), sw))


def test_padded_gate_columns_are_zero():
    # an 8-expert gate padded to 16 output channels with zero weights: the
    # first 8 columns are the gate's logits, the other 8 are exactly 0
    rng = np.random.default_rng(5)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(finite, size=(6, 32)).astype(np.uint8)
    gate = rng.choice(finite, size=(8, 32)).astype(np.uint8)
    padded = np.concatenate([gate, np.zeros((8, 32), np.uint8)])
    y = oracle.scaled_mm_bruteforce(qa, padded, np.float32(0.5), [np.float32(0.25)])
    assert np.array_equal(y[:, :8], oracle.scaled_mm_bruteforce(qa, gate, np.float32(0.5),
                                                                  [np.float32(0.25)]))
    assert np.all(y[:, 8:] == 0)
