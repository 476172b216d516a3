"""Selected embedding rows and the merged LoRA weight of an NF4 base: plain CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Two more consumers of the NF4 format, from [ADAPT] "Native model adaptation and NF4":

* section "Packed NF4 and the portable QLoRA profile": an embedding decodes only the
  rows it selects; section "Fused GPU NF4 decodes inside the matrix kernel": the
  selected-row embedding kernels decode the NF4 codes and the optional nested dynamic8
  scales on the device.  With E = deq(E_nf4) viewed as [rows, dim]:

      out[i][d] = E[ids[i]][d]

  Each element is decoded on its own from the stored bytes, exactly as
  ``nf4.dequantize`` decodes it (w_e = nf4[q_e] * a'_b, b = e // 64, e = id*dim + d);
  an id outside [0, rows) is an error: its row is zeros and the call reports it.

* section "Checkpoints, exact continuation and deployment": export writes merged F32
  deployment weights that include the decoded NF4 base, one matrix at a time.  With
  the adapter of the linear (y = x W^T + s x A^T B^T):

      W' = deq(W) + s B A          [N, K],  A [r, K], B [N, r]

  so that x W'^T equals the adapted linear's output.  Computed here in float64 from
  the float32 decoded base and the float32 adapter.

Pins: tests/test_oracle_export.py (exactly representable tables, a permutation of
rows, the out-of-range row, B = 0, an integer case computed by hand, the rank-1
closed form, and x W'^T against the forward oracle).
"""

import numpy as np

from .codebooks import dynamic8_codebook, nf4_codebook
from .nf4 import BLOCK, NESTED_BLOCK


def _element(qt: dict, e: int, nf4: np.ndarray, dyn8: np.ndarray) -> np.float32:
    """Decoded value of flat element e: nf4[q_e] * a'_b in float32 (a' with two roundings)."""
    byte = int(qt["packed"][e // 2])
    q = (byte & 15) if (e % 2) else (byte >> 4)
    b = e // BLOCK
    if qt["double_quant"]:
        prod = np.float32(dyn8[int(qt["absmax"][b])] * np.float32(qt["nested"][b // NESTED_BLOCK]))
        scale = np.float32(prod + np.float32(qt["offset"]))
    else:
        scale = np.float32(qt["absmax"][b])
    return np.float32(nf4[q] * scale)


def embedding_rows(qt: dict, rows: int, dim: int, ids) -> tuple:
    """(out [len(ids), dim] float32, bad) -- the decoded rows ids of the table qt [rows, dim].

    bad is True when some id lies outside [0, rows); those rows are zeros.  Decodes
    element by element (pure Python: keep the selection small).
    """
    if qt["numel"] != rows * dim:
        raise ValueError("table size does not match rows * dim")
    nf4 = nf4_codebook()
    dyn8 = dynamic8_codebook()
    ids = [int(i) for i in ids]
    out = np.zeros((len(ids), dim), dtype=np.float32)
    bad = False
    for i, r in enumerate(ids):
        if r < 0 or r >= rows:
            bad = True
            continue
        for d in range(dim):
            out[i, d] = _element(qt, r * dim + d, nf4, dyn8)
    return out, bad


def decoded_elements(qt: dict, flat_index) -> np.ndarray:
    """Decoded float32 values of the given flat elements (for sampling large tensors)."""
    nf4 = nf4_codebook()
    dyn8 = dynamic8_codebook()
    return np.array([_element(qt, int(e), nf4, dyn8) for e in np.ravel(flat_index)], dtype=np.float32)


def merge(w_dec: np.ndarray, A: np.ndarray, B: np.ndarray, s: float) -> np.ndarray:
    """W' = W + s B A in float64 from the decoded float32 base W [N, K] and A [r, K], B [N, r]."""
    W = np.asarray(w_dec, dtype=np.float32).astype(np.float64)
    A64 = np.asarray(A, dtype=np.float32).astype(np.float64)
    B64 = np.asarray(B, dtype=np.float32).astype(np.float64)
    if W.shape != (B64.shape[0], A64.shape[1]) or A64.shape[0] != B64.shape[1]:
        raise ValueError("shapes do not match: W [N, K], A [r, K], B [N, r]")
    return W + float(s) * (B64 @ A64)


def merge_entries(w_dec_entries, A: np.ndarray, B: np.ndarray, s: float, n_idx, k_idx) -> np.ndarray:
    """W'[n][k] at the given (n, k) pairs, each one from its own dot product (for sampling)."""
    A64 = np.asarray(A, dtype=np.float32).astype(np.float64)
    B64 = np.asarray(B, dtype=np.float32).astype(np.float64)
    n_idx = np.asarray(n_idx)
    k_idx = np.asarray(k_idx)
    d = np.einsum("ij,ji->i", B64[n_idx, :], A64[:, k_idx])
    return np.asarray(w_dec_entries, dtype=np.float32).astype(np.float64) + float(s) * d
