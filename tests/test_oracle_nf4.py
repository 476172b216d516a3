"""Pins for the oracle's NF4 quantize / dequantize (CPU only).

Each test ties the oracle to something other than itself: the byte counts the pages
print, hand-derived bytes for a block built from code values, exact rational
arithmetic, the round-trip error bound, and invariants of the format.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codebooks as cb
from oracle import nf4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NF4 = cb.nf4_codebook()
DYN8 = cb.dynamic8_codebook()


def _read_byte_counts():
    shapes, totals = [], {}
    with open(os.path.join(GOLDEN, "byte_counts.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) == 3:
                shapes.append(tuple(int(p) for p in parts))
            else:
                totals[parts[0]] = int(parts[1])
    return shapes, totals


def test_byte_formula_matches_printed_per_matrix_counts():
    shapes, _ = _read_byte_counts()
    assert len(shapes) == 4
    for rows, cols, want in shapes:
        assert nf4.packed_bytes(rows * cols, double_quant=True) == want


def test_byte_formula_matches_printed_model_totals():
    _, totals = _read_byte_counts()
    h, inter, vocab, layers = 576, 1536, 49152, 30
    per_layer = [(576, 576), (192, 576), (192, 576), (576, 576),
                 (inter, h), (inter, h), (h, inter)]
    mats = per_layer * layers + [(vocab, h)]
    assert len(mats) == 211
    packed = sum(nf4.packed_bytes(n * k, True, with_offset=True) for n, k in mats)
    norms = (2 * layers + 1) * h * 4
    assert packed == totals["packed_base_bytes"]
    assert norms == totals["floating_base_bytes"]
    assert packed + norms == totals["weight_bytes"]
    # about 0.516 bytes per parameter ([GATE] "P3 is solved")
    n = 4096 * 14336
    assert abs(nf4.packed_bytes(n, True, True) / n - 0.516) < 1e-3


@pytest.mark.parametrize("rows,cols", [(576, 576), (1536, 576), (3, 100)])
def test_quantized_arrays_have_formula_sizes(rows, cols):
    x = np.random.default_rng(5).standard_normal(rows * cols).astype(np.float32)
    q = nf4.quantize(x, double_quant=True)
    got = q["packed"].size + q["absmax"].size + 4 * q["nested"].size
    assert got == nf4.packed_bytes(rows * cols, True)
    q2 = nf4.quantize(x, double_quant=False)
    assert q2["packed"].size + 4 * q2["absmax"].size == nf4.packed_bytes(rows * cols, False)


def test_hand_derived_block_bytes():
    # absmax 2: -2 -> v=-1 -> code 0; 2 -> code 15; 2*(c8/2) is an exact tie between
    # code 7 (0.0) and code 8 -> lower (7); 2*c13 -> 13; zeros -> 7.
    # Element 2i is the high nibble: bytes 0x0F, 0x7D, then 0x77.
    x = np.zeros(64, dtype=np.float32)
    x[0], x[1] = -2.0, 2.0
    x[2] = np.float32(2.0) * (NF4[8] / np.float32(2.0))
    x[3] = np.float32(2.0) * NF4[13]
    q = nf4.quantize(x, double_quant=False)
    assert q["absmax"].tolist() == [2.0]
    assert q["packed"][:2].tolist() == [0x0F, 0x7D]
    assert set(q["packed"][2:].tolist()) == {0x77}


def test_every_code_value_maps_to_its_index():
    a = np.float32(0.25)                        # power of two: c_k * a is exact
    x = np.zeros(64, dtype=np.float32)
    x[:16] = NF4 * a
    q = nf4.quantize(x, double_quant=False)
    codes = nf4.unpack_codes(q["packed"], 64)
    assert codes[:16].tolist() == list(range(16))
    w = nf4.dequantize(q)
    assert np.array_equal(w[:16], x[:16])


def _exact_float32_midpoints(table):
    mids = []
    for j in range(len(table) - 1):
        m = (Fraction(float(table[j])) + Fraction(float(table[j + 1]))) / 2
        if Fraction(float(np.float32(float(m)))) == m:
            mids.append((j, np.float32(float(m))))
    return mids


def test_exact_ties_go_to_lower_code():
    mids = _exact_float32_midpoints(NF4)
    assert len(mids) >= 3
    x = np.zeros(64, dtype=np.float32)
    x[0] = 1.0                                   # absmax 1: v = x exactly
    for i, (_, m) in enumerate(mids):
        x[1 + i] = m
    q = nf4.quantize(x, double_quant=False)
    codes = nf4.unpack_codes(q["packed"], 64)
    for i, (j, _) in enumerate(mids):
        assert codes[1 + i] == j


def _nearest_exact(v, table):
    """Brute force with rationals: smallest |v - t|, first index on ties."""
    fv = Fraction(float(v))
    best, best_d = None, None
    for i, t in enumerate(table):
        d = abs(fv - Fraction(float(t)))
        if best_d is None or d < best_d:
            best, best_d = i, d
    return best


def test_nearest_code_against_rational_brute_force():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.uniform(-1, 1, 300).astype(np.float32),
                        np.array([m for _, m in _exact_float32_midpoints(NF4)], np.float32),
                        np.array([0.0, -0.0, 1e-45, -1e-45, 1.0, -1.0], np.float32)])
    got = nf4.nearest_code(v, NF4)
    want = [_nearest_exact(t, NF4) for t in v]
    assert got.tolist() == want
    vd = rng.uniform(-1, 1, 200).astype(np.float32)
    vd = np.concatenate([vd, DYN8[:5], np.array([m for _, m in _exact_float32_midpoints(DYN8)][:40],
                                                  np.float32)])
    assert nf4.nearest_code(vd, DYN8).tolist() == [_nearest_exact(t, DYN8) for t in vd]


def test_block_absmax_and_partial_tail():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(64 * 3 + 7) * 0.02).astype(np.float32)
    x[64 * 3 + 2] = -0.5                          # tail block max sits in the short block
    q = nf4.quantize(x, double_quant=False)
    assert q["absmax"].size == 4
    for b in range(4):
        assert q["absmax"][b] == np.max(np.abs(x[64 * b:64 * (b + 1)]))
    assert q["absmax"][3] == np.float32(0.5)
    assert q["packed"].size == (x.size + 1) // 2
    assert q["packed"][-1] & 0x0F == 0            # odd count: pad nibble is 0


def test_zero_block_and_negative_zero():
    x = np.zeros(128, dtype=np.float32)
    x[64:] = -0.0
    x[70] = 0.3
    q = nf4.quantize(x, double_quant=False)
    codes = nf4.unpack_codes(q["packed"], 128)
    assert q["absmax"][0] == 0.0
    assert set(codes[:64].tolist()) == {7}
    assert codes[64] == 7 and codes[70] == 15
    w = nf4.dequantize(q)
    assert np.all(w[:64] == 0)


def test_empty_and_nonfinite_rejected():
    with pytest.raises(ValueError):
        nf4.quantize(np.zeros(0, np.float32))
    for bad in (np.nan, np.inf, -np.inf):
        x = np.zeros(100, np.float32)
        x[37] = bad
        with pytest.raises(ValueError):
            nf4.quantize(x)


def test_offset_is_the_rounded_exact_mean():
    rng = np.random.default_rng(7)
    for n in (64 * 300 + 5, 64 * 256 * 3, 64 * 1000):
        x = (rng.standard_t(5, n) * 0.02).astype(np.float32)
        q = nf4.quantize(x, double_quant=True)
        a = nf4.block_absmax(x)
        exact = sum(Fraction(float(t)) for t in a) / len(a)
        assert q["offset"] == np.float32(cb.rn32(exact))


def test_group_sum_tree_order():
    # a sum that float64 rounds differently by order: the tree adds a[i] + a[i+128]
    # first, so 2^53 + 1 + 1 - stays exact only if the two ones meet before 2^53
    a = np.zeros(256, dtype=np.float64)
    a[0], a[1], a[129] = 2.0 ** 53, 1.0, 1.0
    s = nf4.group_sums(a.astype(np.float64))
    # tree: level 128 pairs (1,129) -> 2; then 2^53 + 2 exact
    assert s[0] == 2.0 ** 53 + 2.0


def test_nested_quantization_special_cases():
    # all block maxima equal: centred values are 0, nested absmax 0, decode gives a exactly
    x = np.tile(np.array([0.5] + [0.1] * 63, np.float32), 300)
    q = nf4.quantize(x, double_quant=True)
    zero_code = int(np.flatnonzero(DYN8 == 0)[0])
    assert set(q["absmax"].tolist()) == {zero_code}
    assert np.all(q["nested"] == 0) and q["offset"] == np.float32(0.5)
    assert np.all(nf4.block_scales(q) == np.float32(0.5))
    # the group's largest centred value maps to +1.0 and reconstructs exactly
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(64 * 256) * 0.02).astype(np.float32)
    q = nf4.quantize(x, double_quant=True)
    a = nf4.block_absmax(x)
    c = (a - q["offset"]).astype(np.float32)
    top = int(np.argmax(np.abs(c)))
    if c[top] > 0:
        assert q["absmax"][top] == 255
        assert nf4.block_scales(q)[top] == np.float32(np.float32(q["nested"][0]) + q["offset"])


def test_decode_rounds_product_and_sum_separately():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(64 * 256 * 4) * 0.02).astype(np.float32)
    q = nf4.quantize(x, double_quant=True)
    scales = nf4.block_scales(q)
    na = np.repeat(q["nested"], 256)
    differs = 0
    for b in range(0, q["absmax"].size, 7):
        d, n_, off = float(DYN8[q["absmax"][b]]), float(na[b]), float(q["offset"])
        two_step = cb.rn32(Fraction(cb.rn32(Fraction(d) * Fraction(n_))) + Fraction(off))
        fused = cb.rn32(Fraction(d) * Fraction(n_) + Fraction(off))
        assert scales[b] == np.float32(two_step)
        differs += fused != two_step
    assert differs > 0          # the inputs do exercise the difference from an FMA


def test_round_trip_error_bound():
    rng = np.random.default_rng(13)
    gmax_half = np.float64(np.max(np.diff(NF4.astype(np.float64))) / 2)
    for dq in (False, True):
        for scale in (0.02, 1.0):
            x = (rng.standard_normal(64 * 512 + 33) * scale).astype(np.float32)
            x[rng.choice(x.size, 40, replace=False)] *= 50       # outliers
            q = nf4.quantize(x, double_quant=dq)
            w = nf4.dequantize(q).astype(np.float64)
            a = np.repeat(nf4.block_absmax(x), 64)[:x.size].astype(np.float64)
            ap = np.repeat(nf4.block_scales(q), 64)[:x.size].astype(np.float64)
            ulp = np.spacing(np.abs(x).astype(np.float32)).astype(np.float64)
            bound = gmax_half * a + np.abs(a - ap) + 4 * ulp + 4 * np.spacing(np.float32(1)) * a
            assert np.all(np.abs(x.astype(np.float64) - w) <= bound)
            if not dq:
                assert np.all(ap == a)


def test_requantization_is_deterministic_and_stable():
    rng = np.random.default_rng(17)
    x = (rng.standard_normal(64 * 256 * 2 + 100) * 0.02).astype(np.float32)
    q1 = nf4.quantize(x, True)
    q2 = nf4.quantize(x.copy(), True)
    for k in ("packed", "absmax", "nested"):
        assert np.array_equal(q1[k], q2[k])
    assert q1["offset"] == q2["offset"]
    # without double quant the decoded tensor re-quantizes to the same codes and absmax
    p = nf4.quantize(x, False)
    p2 = nf4.quantize(nf4.dequantize(p), False)
    assert np.array_equal(p["packed"], p2["packed"])
    assert np.array_equal(p["absmax"], p2["absmax"])


def test_bf16_rounding_against_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 3.4e38, 1e-40],
                                 np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(nf4.round_bf16(x), want)


def test_round_f16_hand_values():
    """IEEE binary16: 11 significant bits, ties to even, subnormals down to 2^-24, overflow to inf."""
    cases = [
        (1.0 + 2.0 ** -11, 1.0),                       # halfway between 1 and 1 + 2^-10: even (1)
        (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),       # halfway between 1 + 2^-10 and 1 + 2^-9: even
        (1.0 + 2.0 ** -11 + 2.0 ** -20, 1.0 + 2.0 ** -10),   # just above halfway: up
        (-1.5 - 2.0 ** -12, -1.5),                     # below half an ulp: down in magnitude
        (65504.0, 65504.0),                            # largest finite
        (65519.99, 65504.0),                           # below the overflow threshold
        (65520.0, np.inf),                             # halfway to 2^16: rounds up, overflows
        (2.0 ** -24, 2.0 ** -24),                      # smallest subnormal
        (2.0 ** -25, 0.0),                             # halfway between 0 and 2^-24: even (0)
        (3 * 2.0 ** -26, 2.0 ** -24),                  # above halfway: up
        (2.0 ** -14 + 2.0 ** -25, 2.0 ** -14),         # halfway in the subnormal spacing: even
    ]
    got = nf4.round_f16(np.array([c[0] for c in cases], dtype=np.float32))
    want = np.array([c[1] for c in cases], dtype=np.float32)
    assert np.array_equal(got, want), list(zip(got, want))


def test_dequantize_f16_is_one_rounding_of_the_fp32_decode():
    rng = np.random.default_rng(17)
    x = (rng.standard_normal(64 * 40 + 7) * 0.02).astype(np.float32)
    q = nf4.quantize(x, double_quant=True)
    w32 = nf4.dequantize(q, "f32")
    w16 = nf4.dequantize(q, "f16")
    # every value is a binary16 number within half an ulp (2^-11 relative) of the fp32 decode
    assert np.array_equal(w16.astype(np.float16).astype(np.float32), w16)
    nz = w32 != 0
    assert np.all(np.abs(w16[nz] - w32[nz]) <= np.abs(w32[nz]) * 2.0 ** -11)
    assert np.all(w16[~nz] == 0)
