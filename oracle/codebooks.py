"""The two constant code tables of NF4 double quantization (oracle copy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[ADAPT] section "Packed NF4 and the portable QLoRA profile" says every matrix uses
"the exact 16 value NF4 codebook" and that the block maxima are quantized "with the
signed dynamic8 codebook", following QLoRA and the bitsandbytes codebooks; [GATE]
section "P3 is solved" says both tables are shared constants (16 fp32 and 256 fp32).
Neither page prints the values, so:

* NF4: the 16 values published in the QLoRA paper (Dettmers et al. 2023,
  appendix "NormalFloat 4-bit data type"), held here as float32 literals.  They
  are pinned (tests/test_oracle_codebooks.py) against an independent float64
  construction from the paper's definition: quantiles of N(0, 1), 8 for the
  positive half and 7 for the negative half at probabilities evenly spaced from
  delta down to 1/2 (1/2 itself dropped), an exact zero, all divided by the
  largest magnitude, with delta = 1 - (1/30 + 1/32) / 2.

* dynamic8: built here from the definition of signed dynamic tree quantization
  (Dettmers et al. 2022, "8-bit Optimizers via Block-wise Quantization", section
  "Dynamic Tree Quantization").  A code is a sign bit and 7 more bits: E leading
  zero bits set the decimal exponent 10^-E, a 1 bit ends them, and the remaining
  F = 6 - E bits index one of 2^F equal bins of [0.1, 1]; the code's magnitude is
  that bin's midpoint times 10^-E.  The two codes whose 7 bits are all zero stand
  for 0 and for +1.0 (so the group maximum round-trips exactly; -1.0 is not in
  the table).  Each value is the exact rational rounded once to float32
  (round-to-nearest-even).  Result: 127 negative values, 0, 127 positive values
  below 1, and 1.0 -- 256 distinct, sorted.
"""

from fractions import Fraction

import numpy as np

# QLoRA paper, appendix "NormalFloat 4-bit data type": the NF4 values, ascending.
_NF4_LITERAL = (
    -1.0,
    -0.6961928009986877,
    -0.5250730514526367,
    -0.39491748809814453,
    -0.28444138169288635,
    -0.18477343022823334,
    -0.09105003625154495,
    0.0,
    0.07958029955625534,
    0.16093020141124725,
    0.24611230194568634,
    0.33791524171829224,
    0.44070982933044434,
    0.5626170039176941,
    0.7229568362236023,
    1.0,
)


def nf4_codebook() -> np.ndarray:
    """The 16 NF4 code values as float32, ascending (index 7 is 0.0)."""
    return np.array(_NF4_LITERAL, dtype=np.float32)


def nf4_codebook_from_quantiles() -> np.ndarray:
    """Float64 construction of NF4 from normal quantiles (used only to pin the literal)."""
    from scipy.stats import norm

    delta = 1.0 - (1.0 / 30.0 + 1.0 / 32.0) / 2.0
    positive = norm.ppf(np.linspace(delta, 0.5, 9)[:-1])   # 8 values
    negative = -norm.ppf(np.linspace(delta, 0.5, 8)[:-1])  # 7 values
    values = np.sort(np.concatenate([negative, [0.0], positive]))
    return values / np.max(np.abs(values))


def rn32(q: Fraction) -> float:
    """Round an exact rational to the nearest float32 (ties to even); returns a Python float."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    q = abs(q)
    # exponent e with 2^e <= q < 2^(e+1)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    e = max(e, -126)                      # subnormal range keeps the minimum exponent
    scaled = q * Fraction(2) ** (23 - e)  # 24-bit significand (fewer when subnormal)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return sign * float(m) * 2.0 ** (e - 23)


def dynamic8_exact() -> list:
    """The 256 dynamic8 values as exact rationals, ascending (0 and +1 included)."""
    vals = [Fraction(0), Fraction(1)]
    for e in range(7):          # E leading zeros
        f_bits = 6 - e
        bins = 2 ** f_bits
        for f in range(bins):
            mid = Fraction(1, 10) + Fraction(2 * f + 1, 2) * Fraction(9, 10) / bins
            mag = mid / Fraction(10) ** e
            vals.append(mag)
            vals.append(-mag)
    vals.sort()
    return vals


def dynamic8_codebook() -> np.ndarray:
    """The 256 dynamic8 code values as float32, ascending."""
    return np.array([rn32(v) for v in dynamic8_exact()], dtype=np.float32)
