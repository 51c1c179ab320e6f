"""Stored fixtures under tests/golden/ (each written by the script beside it):
- e4m3_positive_values.txt, from the FP8 E4M3 definition alone (OCP 8-bit floating point
  specification: bias 7, subnormals m/8 * 2^-6, no infinities, 0x7F NaN, max 448): the
  oracle's decoder must give every value exactly and its encoder must map each value back to
  its code;
- oracle_small_case.txt, the oracle's outputs for one small fully specified case: a change to
  the oracle's arithmetic shows up here (to within float64 summation-order noise)."""

import os
import sys
from fractions import Fraction

import numpy as np

from oracle.fp8 import e4m3_decode, e4m3_encode

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_e4m3_table_from_the_definition():
    rows = _lines("e4m3_positive_values.txt")
    assert len(rows) == 127
    codes = np.array([int(c, 16) for c, _ in rows], dtype=np.uint8)
    vals = np.array([float(Fraction(v)) for _, v in rows])
    np.testing.assert_array_equal(e4m3_decode(codes), vals)
    np.testing.assert_array_equal(e4m3_decode(codes | 0x80), -vals)
    np.testing.assert_array_equal(e4m3_encode(vals), codes)
    assert vals.max() == 448.0 and np.isnan(e4m3_decode(np.array([0x7F], np.uint8)))[0]


def test_oracle_small_case_unchanged():
    sys.path.insert(0, GOLDEN)
    import make_oracle_case
    got = make_oracle_case.compute()
    want_o, want_lse = {}, {}
    for row in _lines("oracle_small_case.txt"):
        causal, r = bool(int(row[1])), int(row[2])
        if row[0] == "o":
            want_o[(causal, r)] = [float.fromhex(x) for x in row[3:]]
        else:
            want_lse[(causal, r)] = float.fromhex(row[3])
    for causal, (o, lse) in got.items():
        for r in range(o.shape[0]):
            np.testing.assert_allclose(o[r], want_o[(causal, r)], rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(lse[r], want_lse[(causal, r)], rtol=1e-12, atol=1e-15)
