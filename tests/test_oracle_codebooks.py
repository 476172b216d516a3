"""Pins for the oracle's two code tables (CPU only).

NF4: the float32 literals are checked against an independent float64 construction
from normal quantiles (QLoRA paper definition) and against structural facts.
dynamic8: the enumerated table is checked against an independent decode of every
8-bit pattern of the dynamic tree format, and against structural facts.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import codebooks as cb


def test_nf4_literal_matches_quantile_construction():
    lit = cb.nf4_codebook().astype(np.float64)
    built = cb.nf4_codebook_from_quantiles()
    assert lit.shape == (16,)
    assert np.max(np.abs(lit - built)) < 1e-6


def test_nf4_structure():
    t = cb.nf4_codebook()
    assert t.dtype == np.float32
    assert np.all(np.diff(t) > 0)
    assert t[0] == -1.0 and t[15] == 1.0 and t[7] == 0.0
    assert np.sum(t < 0) == 7 and np.sum(t > 0) == 8
    gaps = np.diff(t.astype(np.float64))
    # the largest gap sits between -1 and the next code; half of it bounds the
    # normalised rounding error (about 0.1519)
    assert int(np.argmax(gaps)) == 0
    assert abs(gaps.max() / 2 - 0.1519036) < 1e-6


def _decode_dynamic_tree_byte(code: int) -> Fraction:
    """Independent decode of one signed dynamic-tree byte: sign, zeros, indicator, fraction."""
    sign = -1 if code & 0x80 else 1
    rest = code & 0x7F
    if rest == 0:
        # the two all-zero patterns stand for 0 and +1
        return Fraction(0) if sign > 0 else Fraction(1)
    zeros = 0
    bit = 6
    while not (rest >> bit) & 1:
        zeros += 1
        bit -= 1
    frac_bits = bit                      # bits after the indicator
    f = rest & ((1 << frac_bits) - 1)
    lo = Fraction(1, 10) + Fraction(9, 10) * Fraction(f, 1 << frac_bits)
    hi = Fraction(1, 10) + Fraction(9, 10) * Fraction(f + 1, 1 << frac_bits)
    return sign * (lo + hi) / 2 / Fraction(10) ** zeros


def test_dynamic8_matches_bitwise_decode():
    decoded = sorted(_decode_dynamic_tree_byte(c) for c in range(256))
    enumerated = cb.dynamic8_exact()
    assert decoded == enumerated
    t = cb.dynamic8_codebook()
    assert [cb.rn32(v) for v in decoded] == t.tolist()


def test_dynamic8_structure():
    t = cb.dynamic8_codebook()
    assert t.dtype == np.float32 and t.shape == (256,)
    assert np.all(np.diff(t) > 0)               # sorted and distinct
    assert t[-1] == 1.0 and 0.0 in t
    assert t[0] > -1.0                           # -1 is not representable
    assert np.sum(t < 0) == 127 and np.sum((t > 0) & (t < 1)) == 127
    # largest magnitude below 1: midpoint of the top bin of [0.1, 1] split in 64
    assert t[-2] == np.float32(0.1 + 63.5 * 0.9 / 64)
    # smallest positive: the single bin of [0.1, 1] at 10^-6
    assert t[t > 0][0] == np.float32(0.55e-6)
    # decade counts: 64, 32, ..., 1 positive values with magnitude in [0.1, 1) * 10^-E
    pos = t[(t > 0) & (t < 1)].astype(np.float64)
    for e in range(7):
        n = np.sum((pos >= 0.1 * 10.0 ** -e) & (pos < 10.0 ** -e))
        assert n == 2 ** (6 - e)


@pytest.mark.parametrize("q", [Fraction(1, 3), Fraction(-7, 10), Fraction(1, 10 ** 40),
                               Fraction(2 ** 24 + 1, 2 ** 24), Fraction(2 ** 24 + 3, 2 ** 24)])
def test_rn32_agrees_with_numpy_rounding(q):
    # these cases are held exactly by float64 or sit far from a float32 tie, so
    # numpy's float64 -> float32 conversion is a valid reference
    assert np.float32(cb.rn32(q)) == np.float32(float(q))


def test_rn32_ties_to_even():
    # 1 + 2^-24 is halfway between 1 and 1 + 2^-23: ties to the even significand (1.0)
    assert cb.rn32(Fraction(2 ** 24 + 1, 2 ** 24)) == 1.0
    # 1 + 3*2^-24 is halfway between 1 + 2^-23 and 1 + 2^-22: goes to 1 + 2^-22
    assert cb.rn32(Fraction(2 ** 24 + 3, 2 ** 24)) == 1.0 + 2.0 ** -22
