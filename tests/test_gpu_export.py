"""GPU parity of the selected-row embedding decode and the merged LoRA weight (C ABI).

Embedding rows are bit-exact against the oracle (fp32 values, and their bfloat16
rounding).  The merged weight is compared with the oracle's float64 W + s B A within
the bound of its fp32 arithmetic: the rank-r dot product by fused multiply-adds
(r roundings), s * d and w + s * d (one rounding each) give

    |W'_gpu - W'| <= u |W'| + (r + 2) u |s| sum_j |B[n][j] A[j][k]|,   u = 2^-24,

and a bfloat16 output adds its own rounding, 2^-8 |W'|.  Inputs come from the
seeded generators in bit_nf4_quantized_gb300.workloads.
"""

import numpy as np
import pytest
import torch

from bit_nf4_quantized_gb300 import binding
from bit_nf4_quantized_gb300 import workloads as wl
from oracle import export as oexp
from oracle import nf4 as onf4

pytestmark = pytest.mark.gpu

DEV = "cuda"
U32 = 2.0 ** -24


def _upload(ref, shape):
    """A stored NF4 tensor (oracle output or random bytes) copied to the device."""
    q = binding.Nf4Tensor.empty(shape, ref["double_quant"], DEV)
    q.packed.copy_(torch.from_numpy(ref["packed"]))
    q.absmax.copy_(torch.from_numpy(ref["absmax"]))
    if ref["double_quant"]:
        q.nested_absmax.copy_(torch.from_numpy(ref["nested"]))
        q.offset[0] = float(ref["offset"])
    return q


def _random_stored(shape, dq, workload, tensor_id):
    n = int(np.prod(shape))
    parts = wl.random_nf4_parts((n + 1) // 2, onf4.num_blocks(n), onf4.num_nested(n), dq, workload, tensor_id)
    parts.update(numel=n, double_quant=dq)
    return parts


def _f32_bits(t):
    return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ---- selected embedding rows --------------------------------------------------------

EMB_SHAPES = [(40, 64), (37, 100), (9, 4160), (5, 2049), (3, 7), (300, 8), (30, 576)]


@pytest.mark.parametrize("rows,dim", EMB_SHAPES)
@pytest.mark.parametrize("dq", [True, False])
def test_embedding_rows_bit_exact(lib, rows, dim, dq):
    x = wl.student_t(rows * dim, 5, 0.02, 6, 1)
    ref = onf4.quantize(x, double_quant=dq)
    E = _upload(ref, (rows, dim))
    ids_np = wl.token_ids(12, rows, 6, 2)
    ids_np[1], ids_np[3], ids_np[-1] = 0, ids_np[0], rows - 1     # first, repeated, last row
    want, bad = oexp.embedding_rows(ref, rows, dim, ids_np)
    assert not bad
    ids = torch.from_numpy(ids_np).to(DEV)
    binding.device_status(clear=True)
    got = binding.nf4_embedding_rows(E, ids, torch.float32)
    got_bf = binding.nf4_embedding_rows(E, ids, torch.bfloat16)
    assert binding.device_status(clear=True) == binding.NF4_OK
    assert np.array_equal(_f32_bits(got), want.view(np.uint32))
    assert np.array_equal(_bf16_bits(got_bf), onf4.bf16_bits(onf4.round_bf16(want)))


@pytest.mark.parametrize("dim", [200, 256])
def test_embedding_out_of_range_ids(lib, dim):
    rows = 20
    ref = onf4.quantize(wl.normal(rows * dim, 0.02, 6, 3), double_quant=True)
    E = _upload(ref, (rows, dim))
    ids_np = np.array([1, rows, -5, 19, 1 << 40], dtype=np.int64)
    want, bad = oexp.embedding_rows(ref, rows, dim, ids_np)
    assert bad
    binding.device_status(clear=True)
    out = torch.full((5, dim), 7.0, device=DEV)                    # zeros must be written
    binding.nf4_embedding_rows(E, torch.from_numpy(ids_np).to(DEV), out=out)
    assert binding.device_status(clear=True) == binding.NF4_ERR_ARG
    assert np.array_equal(_f32_bits(out), want.view(np.uint32))
    assert not out[[1, 2, 4]].any()
    binding.nf4_embedding_rows(E, torch.tensor([0, 19], device=DEV))
    assert binding.device_status(clear=True) == binding.NF4_OK


@pytest.mark.parametrize("dim", [96, 100])
def test_embedding_more_ids_than_resident_warps(lib, dim):
    """6000 ids: each warp of the row-per-warp kernel takes several rows."""
    rows = 50
    ref = onf4.quantize(wl.normal(rows * dim, 0.02, 6, 5), double_quant=True)
    E = _upload(ref, (rows, dim))
    ids_np = wl.token_ids(6000, rows, 6, 6)
    ids = torch.from_numpy(ids_np).to(DEV)
    full = binding.nf4_dequantize(E, torch.float32)
    for dtype in (torch.float32, torch.bfloat16):
        got = binding.nf4_embedding_rows(E, ids, dtype)
        assert torch.equal(got.view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                           full[ids].to(dtype).view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    pick = [0, 1, 2999, 5999]
    want, _ = oexp.embedding_rows(ref, rows, dim, ids_np[pick])
    assert np.array_equal(_f32_bits(binding.nf4_embedding_rows(E, ids, torch.float32)[pick]), want.view(np.uint32))
    assert binding.device_status(clear=True) == binding.NF4_OK


def test_embedding_no_ids_launches_nothing(lib):
    ref = onf4.quantize(wl.normal(64 * 10, 0.02, 6, 4), double_quant=True)
    E = _upload(ref, (10, 64))
    before = binding.launch_count()
    out = binding.nf4_embedding_rows(E, torch.empty(0, dtype=torch.int64, device=DEV))
    assert out.shape == (0, 64)
    assert binding.launch_count() == before


def test_embedding_full_table_sampled(lib):
    """128256 x 4096 table of random stored bytes, 4096 ids (the measured case)."""
    w = wl.W6
    rows, dim, n_ids = w["rows"], w["dim"], w["n_ids"]
    stored = _random_stored((rows, dim), True, 6, 10)
    E = _upload(stored, (rows, dim))
    ids_np = wl.token_ids(n_ids, rows, 6, 11)
    ids = torch.from_numpy(ids_np).to(DEV)
    binding.device_status(clear=True)
    got_bf = binding.nf4_embedding_rows(E, ids, torch.bfloat16)
    got = binding.nf4_embedding_rows(E, ids, torch.float32)
    assert binding.device_status(clear=True) == binding.NF4_OK
    # every row: the bits that dequantize writes for the same elements
    full = binding.nf4_dequantize(E, torch.float32).view(rows, dim)
    assert torch.equal(got.view(torch.int32), full[ids].view(torch.int32))
    del full
    # sampled rows, element by element, against the oracle
    pick = np.array([0, 1, n_ids // 2, n_ids - 1] + list(wl.rng(6, 12).integers(0, n_ids, size=4)))
    flat = (ids_np[pick][:, None] * dim + np.arange(dim)[None, :]).ravel()
    want = oexp.decoded_elements(stored, flat).reshape(len(pick), dim)
    assert np.array_equal(_f32_bits(got[torch.from_numpy(pick).to(DEV)]), want.view(np.uint32))
    assert np.array_equal(_bf16_bits(got_bf[torch.from_numpy(pick).to(DEV)]),
                          onf4.bf16_bits(onf4.round_bf16(want)))


# ---- merged weight ------------------------------------------------------------------

def _merge_bound(ref, A, B, s, r, bf16):
    S = abs(s) * (np.abs(B.astype(np.float64)) @ np.abs(A.astype(np.float64)))
    tol = U32 * np.abs(ref) + (r + 2) * U32 * S * 1.01
    if bf16:
        tol = tol + 2.0 ** -8 * (np.abs(ref) + tol)
    return tol


def _s32(alpha, r, mode):
    if mode == binding.SCALE_LORA:
        return float(np.float32(alpha) / np.float32(r))
    return float(np.float32(float(alpha) / np.sqrt(float(r))))


# (8, 80000, 4): 313 column tiles, more than the resident CTAs, so a CTA's tiles change
# column range and A is restaged per tile
MERGE_CASES = [(64, 256, 16), (200, 520, 17), (7, 8, 1), (130, 264, 64), (300, 512, 256), (72, 1024, 5),
               (8, 80000, 4)]


@pytest.mark.parametrize("N,K,r", MERGE_CASES)
@pytest.mark.parametrize("dq", [True, False])
def test_merge_lora_matches_oracle(lib, N, K, r, dq):
    ref_q = onf4.quantize(wl.student_t(N * K, 5, 0.02, 7, 1), double_quant=dq)
    W = _upload(ref_q, (N, K))
    A = wl.normal((r, K), 1.0 / np.sqrt(r), 7, 2)
    B = wl.normal((N, r), 0.02, 7, 3)
    mode = binding.SCALE_RSLORA if r == 17 else binding.SCALE_LORA
    alpha = 16.0 if r != 5 else 12.0                            # 12 / 5 is not exact in fp32
    s = _s32(alpha, r, mode)
    want = oexp.merge(onf4.dequantize(ref_q).reshape(N, K), A, B, s)
    Ad, Bd = torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)
    got = binding.nf4_merge_lora(W, Ad, Bd, alpha, mode, torch.float32)
    got_bf = binding.nf4_merge_lora(W, Ad, Bd, alpha, mode, torch.bfloat16)
    g64 = got.cpu().numpy().astype(np.float64)
    err = np.abs(g64 - want)
    assert np.all(err <= _merge_bound(want, A, B, s, r, False)), float(err.max())
    gb = got_bf.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gb - want) <= _merge_bound(want, A, B, s, r, True))
    # the bf16 output is the fp32 merged value rounded once
    assert np.array_equal(_bf16_bits(got_bf), onf4.bf16_bits(onf4.round_bf16(got.cpu().numpy())))


def test_merge_zero_adapter_is_dequantize(lib):
    N, K, r = 96, 320, 8
    ref_q = onf4.quantize(wl.normal(N * K, 0.02, 7, 5), double_quant=True)
    W = _upload(ref_q, (N, K))
    A = torch.from_numpy(wl.normal((r, K), 0.3, 7, 6)).to(DEV)
    B = torch.zeros((N, r), device=DEV)
    got = binding.nf4_merge_lora(W, A, B, 16.0)
    # equal values (w + s * 0 turns a -0 weight into +0; every other value keeps its bits)
    assert np.array_equal(got.cpu().numpy().ravel(), onf4.dequantize(ref_q))


def test_merge_full_gate_matrix_sampled(lib):
    """14336 x 4096, r = 16 (the measured case): sampled entries and whole rows."""
    w = wl.W7
    N, K, r, alpha = w["N"], w["K"], w["r"], w["alpha"]
    stored = _random_stored((N, K), True, 7, 20)
    W = _upload(stored, (N, K))
    A, B = wl.adapters(N, K, r, 7, 21)
    s = _s32(alpha, r, binding.SCALE_LORA)
    got = binding.nf4_merge_lora(W, torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV), alpha)
    got_bf = binding.nf4_merge_lora(W, torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV), alpha,
                                    dtype=torch.bfloat16)
    g = wl.rng(7, 22)
    n_idx = np.concatenate([g.integers(0, N, size=4096), np.repeat([0, N - 1, 7777], K)])
    k_idx = np.concatenate([g.integers(0, K, size=4096), np.tile(np.arange(K), 3)])
    flat = n_idx.astype(np.int64) * K + k_idx
    want = oexp.merge_entries(oexp.decoded_elements(stored, flat), A, B, s, n_idx, k_idx)
    gv = got.view(-1)[torch.from_numpy(flat).to(DEV)].cpu().numpy().astype(np.float64)
    S = abs(s) * np.einsum("ij,ji->i", np.abs(B[n_idx].astype(np.float64)), np.abs(A[:, k_idx].astype(np.float64)))
    tol = U32 * np.abs(want) + (r + 2) * U32 * S * 1.01
    assert np.all(np.abs(gv - want) <= tol)
    # at full size: the bf16 output is the fp32 output rounded once
    assert torch.equal(got_bf.view(torch.int16), got.to(torch.bfloat16).view(torch.int16))
