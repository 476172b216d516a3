"""Pins for the oracle's selected embedding rows and merged LoRA weight (CPU only).

Embedding rows: tables whose every value the format stores exactly (so decoding the
selected rows must give the original numbers back), a hand-built double-quantized
table whose scales are exact (dynamic8 codes 0 and +1, two nested groups), the
out-of-range row, and agreement with the vectorised dequantize on a ragged shape.
Merge: B = 0, an integer case worked by hand, the rank-1 closed form, and
x W'^T against the forward oracle of the adapted linear.
"""

import numpy as np
import pytest

from oracle import codebooks, export, nf4, qlora

NF4 = codebooks.nf4_codebook()
DYN8 = codebooks.dynamic8_codebook()


def _exact_table(rows, dim, seed):
    """Values nf4[q] * 2^e, every 64-block holding +1 or -1 times its 2^e (absmax = 2^e)."""
    rng = np.random.default_rng(seed)
    n = rows * dim
    q = rng.integers(0, 16, size=n)
    nb = -(-n // 64)
    e = rng.integers(-6, 4, size=nb)
    for b in range(nb):
        q[b * 64 + rng.integers(0, min(64, n - b * 64))] = rng.choice([0, 15])
    x = (NF4[q] * np.ldexp(np.float32(1.0), np.repeat(e, 64)[:n]).astype(np.float32)).astype(np.float32)
    return x.reshape(rows, dim)


@pytest.mark.parametrize("rows,dim", [(9, 64), (7, 100), (5, 33)])
def test_embedding_returns_exactly_stored_rows(rows, dim):
    x = _exact_table(rows, dim, seed=rows * dim)
    qt = nf4.quantize(x, double_quant=False)
    ids = [3, 0, rows - 1, 3, 1]
    out, bad = export.embedding_rows(qt, rows, dim, ids)
    assert not bad
    assert np.array_equal(out, x[ids])


def test_embedding_hand_built_double_quant_scales():
    # 2 nested groups (512 blocks of 64 = 32768 elements, [16, 2048]).  Absmax code
    # 127 is dynamic8 0.0 -> a' = offset = 0.5; code 255 is +1.0 -> a' = na + offset,
    # 0.5 + 0.5 = 1 in group 0 and 1.5 + 0.5 = 2 in group 1.  Every product is exact.
    assert DYN8[127] == 0.0 and DYN8[255] == 1.0
    rows, dim = 16, 2048
    n = rows * dim
    rng = np.random.default_rng(11)
    q = rng.integers(0, 16, size=n).astype(np.uint8)
    codes = rng.choice(np.array([127, 255], dtype=np.uint8), size=n // 64)
    qt = dict(numel=n, double_quant=True, packed=((q[0::2] << 4) | q[1::2]).astype(np.uint8),
              absmax=codes, nested=np.array([0.5, 1.5], dtype=np.float32), offset=np.float32(0.5))
    scale_of_block = np.where(codes == 127, 0.5, np.where(np.arange(n // 64) < 256, 1.0, 2.0))
    want = (NF4[q].astype(np.float64) * np.repeat(scale_of_block, 64)).reshape(rows, dim)
    ids = [15, 0, 8, 7]
    out, bad = export.embedding_rows(qt, rows, dim, ids)
    assert not bad
    assert np.array_equal(out.astype(np.float64), want[ids])


def test_embedding_out_of_range_id_gives_zero_row_and_flag():
    x = _exact_table(4, 64, seed=3)
    qt = nf4.quantize(x, double_quant=False)
    out, bad = export.embedding_rows(qt, 4, 64, [1, 4, -1, 2])
    assert bad
    assert np.array_equal(out[[0, 3]], x[[1, 2]])
    assert not out[[1, 2]].any()


@pytest.mark.parametrize("dq", [True, False])
def test_embedding_all_rows_equals_dequantize(dq):
    rows, dim = 6, 150                                    # blocks straddle rows; odd tail
    x = np.random.default_rng(9).standard_normal(rows * dim).astype(np.float32)
    qt = nf4.quantize(x, double_quant=dq)
    out, bad = export.embedding_rows(qt, rows, dim, range(rows))
    assert not bad
    full = nf4.dequantize(qt).reshape(rows, dim)
    assert np.array_equal(out.view(np.uint32), full.view(np.uint32))
    perm = [5, 2, 0, 4, 1, 3]
    out2, _ = export.embedding_rows(qt, rows, dim, perm)
    assert np.array_equal(out2, full[perm])


def test_merge_with_zero_b_is_the_decoded_base():
    rng = np.random.default_rng(2)
    W = rng.standard_normal((6, 16)).astype(np.float32)
    A = rng.standard_normal((3, 16)).astype(np.float32)
    out = export.merge(W, A, np.zeros((6, 3), np.float32), 1.7)
    assert np.array_equal(out, W.astype(np.float64))


def test_merge_integer_case_by_hand():
    # B A = [[1*1 + 2*0, 1*0 + 2*1, 1*2 + 2*(-1)], [3*1 - 1*0, 3*0 - 1*1, 3*2 - 1*(-1)]]
    #     = [[1, 2, 0], [3, -1, 7]];  W + 0.5 B A with W = [[1, 1, 1], [0, 0, 0]]
    W = np.array([[1, 1, 1], [0, 0, 0]], np.float32)
    A = np.array([[1, 0, 2], [0, 1, -1]], np.float32)
    B = np.array([[1, 2], [3, -1]], np.float32)
    want = np.array([[1.5, 2.0, 1.0], [1.5, -0.5, 3.5]])
    assert np.array_equal(export.merge(W, A, B, 0.5), want)


def test_merge_rank_one_is_an_outer_product():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((5, 8)).astype(np.float32)
    a = rng.standard_normal(8).astype(np.float32)
    b = rng.standard_normal(5).astype(np.float32)
    got = export.merge(W, a[None, :], b[:, None], 2.5)
    for n in range(5):
        for k in range(8):
            want = float(W[n, k]) + 2.5 * float(b[n]) * float(a[k])
            assert got[n, k] == pytest.approx(want, rel=1e-15, abs=1e-15)


def test_merged_weight_reproduces_the_adapted_linear():
    rng = np.random.default_rng(8)
    M, N, K, r = 7, 12, 40, 4
    x = rng.standard_normal((M, K)).astype(np.float32)
    W = nf4.dequantize(nf4.quantize(rng.standard_normal(N * K).astype(np.float32))).reshape(N, K)
    A = rng.standard_normal((r, K)).astype(np.float32)
    B = rng.standard_normal((N, r)).astype(np.float32)
    s = qlora.lora_scale(16.0, r)
    y, _ = qlora.forward(x, W, A, B, s, compute="f32")
    y_merged = x.astype(np.float64) @ export.merge(W, A, B, s).T
    assert np.max(np.abs(y_merged - y)) <= 1e-12 * np.max(np.abs(y))


def test_merge_entries_match_the_full_merge():
    rng = np.random.default_rng(6)
    W = rng.standard_normal((9, 24)).astype(np.float32)
    A = rng.standard_normal((5, 24)).astype(np.float32)
    B = rng.standard_normal((9, 5)).astype(np.float32)
    full = export.merge(W, A, B, 0.75)
    n_idx = np.array([0, 8, 3, 3])
    k_idx = np.array([23, 0, 11, 12])
    part = export.merge_entries(W[n_idx, k_idx], A, B, 0.75, n_idx, k_idx)
    assert np.allclose(part, full[n_idx, k_idx], rtol=1e-15, atol=0)
