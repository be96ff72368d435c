"""Pins of the oracle's parity criteria: the acceptance functions through
which every GPU parity test of a floating-point product passes.

The 16-bit tolerance is the layer specification's: elementwise
1e-2 (|y_ref| + rms(y_ref)) and relative Frobenius 5e-3 against the float64
product of the same E4M3 operands.  The E4M3-output criterion is this
library's reading of it for outputs re-quantized through output_scale ("RFC:
FP8 Quantization Schema in vLLM", the output_scale discussion): one code
step of E4M3(y_ref / output_scale), exact away from rounding midpoints."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def table():
    return oracle.decode_table()


def test_gemm_close():
    pins.check_gemm_close(oracle.gemm_close)


def test_midpoint_distance(table):
    pins.check_midpoint_distance(oracle._nearest_midpoint_distance, table)


def test_e4m3_output_close(table):
    pins.check_e4m3_output_close(oracle.e4m3_output_close, table)
