"""The seeded input generators (CPU): sizes, types, ranges and determinism.

These draw the stored bytes and token ids of the full-size selected-row and merge cases,
so a change in them would silently change what those tests compare.
"""

import numpy as np

from bit_nf4_quantized_gb300 import workloads as wl
from oracle import nf4 as onf4


def test_random_nf4_parts_sizes_and_ranges():
    n = 64 * 256 * 3 + 100
    nb, nnb = onf4.num_blocks(n), onf4.num_nested(n)
    dq = wl.random_nf4_parts((n + 1) // 2, nb, nnb, True, 9, 1)
    assert dq["packed"].dtype == np.uint8 and dq["packed"].size == (n + 1) // 2
    assert dq["absmax"].dtype == np.uint8 and dq["absmax"].size == nb
    assert dq["nested"].dtype == np.float32 and dq["nested"].size == nnb
    assert np.all((dq["nested"] >= 0.01) & (dq["nested"] < 0.05))
    assert dq["offset"] == np.float32(0.03)
    assert dq["packed"].min() < 16 and dq["packed"].max() > 240       # the whole byte range is drawn
    plain = wl.random_nf4_parts((n + 1) // 2, nb, nnb, False, 9, 1)
    assert plain["absmax"].dtype == np.float32 and plain["absmax"].size == nb
    assert np.all(plain["absmax"] > 0) and plain["nested"] is None and plain["offset"] is None


def test_random_nf4_parts_are_seeded():
    a = wl.random_nf4_parts(1000, 32, 1, True, 6, 10)
    b = wl.random_nf4_parts(1000, 32, 1, True, 6, 10)
    c = wl.random_nf4_parts(1000, 32, 1, True, 6, 11)
    assert all(np.array_equal(a[k], b[k]) for k in ("packed", "absmax", "nested"))
    assert not np.array_equal(a["packed"], c["packed"])


def test_token_ids_range_and_seed():
    ids = wl.token_ids(5000, 128256, 6, 11)
    assert ids.dtype == np.int64 and ids.shape == (5000,)
    assert ids.min() >= 0 and ids.max() < 128256
    assert np.array_equal(ids, wl.token_ids(5000, 128256, 6, 11))
    assert len(np.unique(ids)) > 4900                                 # uniform over a large table
