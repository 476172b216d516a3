"""GPU parity of qlora_linear_fwd / qlora_linear_bwd against the float64 oracle.

Every output is checked three ways (tests/parity.py): the stated relative Frobenius
tolerance (1e-5 for the fp32 profile, 2e-2 for the bf16 profile), the same norm over every
256 x 256 block, and an element-wise bound from the magnitudes of the terms of each sum.
Every case uses B != 0 so the adapter path carries weight.
"""

import math

import numpy as np
import pytest
import torch

from bit_nf4_quantized_gb300 import binding
from bit_nf4_quantized_gb300 import workloads as wl
from oracle import nf4 as onf4
from oracle import qlora

import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _quantized_weight(N, K, seed, dist="normal", dq=True):
    if dist == "t":
        w = wl.student_t((N, K), 5, 0.02, 3, seed)
    else:
        w = wl.normal((N, K), 0.02, 2, seed)
    ref = onf4.quantize(w, double_quant=dq)
    q = binding.Nf4Tensor.empty((N, K), dq, DEV)
    q.packed.copy_(torch.from_numpy(ref["packed"]))
    q.absmax.copy_(torch.from_numpy(ref["absmax"]))
    if dq:
        q.nested_absmax.copy_(torch.from_numpy(ref["nested"]))
        q.offset[0] = float(ref["offset"])
    return q, onf4.dequantize(ref, "f32").reshape(N, K)


def _run_case(M, N, K, r, alpha, compute, mode=binding.SCALE_LORA, seed=0, dist="normal", rows=None, dq=True):
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[compute]
    q, w_deq = _quantized_weight(N, K, seed, dist, dq)
    x = wl.normal((M, K), 1.0, 1, seed + 1)
    dy = wl.normal((M, N), 1.0, 1, seed + 2)
    A, B = wl.adapters(N, K, r, 1, seed + 3)
    xd = torch.from_numpy(x).to(DEV).to(tdt)
    dyd = torch.from_numpy(dy).to(DEV).to(tdt)
    Ad, Bd = torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)
    y, T = binding.qlora_linear_fwd(xd, q, Ad, Bd, alpha, mode)
    dx, dA, dB = binding.qlora_linear_bwd(dyd, xd, T, q, Ad, Bd, alpha, mode)
    torch.cuda.synchronize()
    s = qlora.lora_scale(alpha, r, "lora" if mode == binding.SCALE_LORA else "rslora")
    xh, dyh = xd.float().cpu().numpy(), dyd.float().cpu().numpy()
    sel = slice(None) if rows is None else rows
    y_ref, T_ref = qlora.forward(xh[sel], w_deq, A, B, s, compute)
    dX_ref, _, _, _ = qlora.backward(dyh[sel], xh[sel], w_deq, A, B, s, compute)
    dA_ref, dB_ref, _ = qlora.adapter_backward(dyh, xh, A, B, s, compute)
    fb = parity.forward_bounds(xh[sel], w_deq, A, B, s, compute, y_ref, T_ref)
    bb = parity.backward_bounds(dyh, xh, None, A, B, s, compute, dA_ref=dA_ref, dB_ref=dB_ref)
    bx = parity.backward_bounds(dyh[sel], xh[sel], w_deq, A, B, s, compute, dX_ref=dX_ref)
    got = dict(y=y.float().cpu().numpy()[sel], T=T.cpu().numpy()[sel], dX=dx.float().cpu().numpy()[sel],
               dA=dA.cpu().numpy(), dB=dB.cpu().numpy())
    want = dict(y=y_ref, T=T_ref, dX=dX_ref, dA=dA_ref, dB=dB_ref)
    bounds = dict(y=fb["y"], T=fb["T"], dX=bx["dX"], dA=bb["dA"], dB=bb["dB"])
    report = parity.check(got, want, bounds, compute)
    assert np.any(got["dA"] != 0)
    return report


def test_fp32_profile_576(lib):
    c = wl.W1
    _run_case(c["M"], c["N"], c["K"], c["r"], c["alpha"], "f32")


@pytest.mark.parametrize("M,N,K,r", [(1, 8, 64, 1), (3, 40, 100, 2), (77, 130, 200, 5), (200, 96, 64, 16)])
def test_fp32_profile_ragged(lib, M, N, K, r):
    _run_case(M, N, K, r, 8.0, "f32", seed=M)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 17, 33])
def test_bf16_small_m(lib, M):
    _run_case(M, 520, 1024, 8, 16.0, "bf16", seed=M)


@pytest.mark.parametrize("M,N,K,r", [(64, 8, 64, 1), (130, 200, 192, 5), (300, 264, 576, 16),
                                     (511, 1032, 640, 64), (129, 136, 128, 128)])
def test_bf16_tiles_and_tails(lib, M, N, K, r):
    _run_case(M, N, K, r, 16.0, "bf16", seed=N)


@pytest.mark.parametrize("compute", ["bf16", "f32"])
@pytest.mark.parametrize("M,N,K,r", [(130, 200, 192, 5), (512, 1536, 576, 16)])
def test_weight_without_double_quant(lib, compute, M, N, K, r):
    """fp32 block maxima instead of dynamic8 codes: the same kernels with the plain scale."""
    if compute == "f32" and (N, K) == (1536, 576):
        M = 64
    _run_case(M, N, K, r, 16.0, compute, seed=41, dq=False)


def test_bf16_rslora_scale(lib):
    _run_case(40, 256, 512, 8, 16.0, "bf16", mode=binding.SCALE_RSLORA)


def test_bf16_rank_256(lib):
    _run_case(96, 512, 256, 256, 16.0, "bf16")


def test_smollm2_qv_shapes(lib):
    c = wl.W2
    for name, N, K in c["shapes"]:
        if name in c["targets"]:
            _run_case(c["M"], N, K, c["r"], c["alpha"], "bf16", seed=N)


@pytest.mark.parametrize("name,M", [("k_proj", 4096), ("gate_proj", 4096), ("down_proj", 4096),
                                    ("gate_proj", 4881), ("down_proj", 4881)])
def test_llama8b_layer_sampled_rows(lib, name, M):
    """The Llama-3-8B-shaped projections at 4096 tokens, and gate and down at 4881 tokens.
    Down's forward and gate's dX have both operands larger than half of L2, so their GEMM
    takes the tile pairs in bands of 8 token tiles; 4881 tokens make 20 token tiles, the last
    band 4 tiles and ragged.  Sampled token rows, always with those at band and tile edges."""
    c = wl.W3
    N, K = {n: (a, b) for n, a, b in c["shapes"]}[name]
    edges = [r for r in (0, 255, 256, 2047, 2048, 4095, 4096, M - 1) if r < M]
    rows = np.unique(np.concatenate([np.random.default_rng(5).choice(M, 64, replace=False), edges]))
    _run_case(M, N, K, c["r"], c["alpha"], "bf16", seed=K, dist="t", rows=rows)


@pytest.mark.parametrize("N,K", [(1344, 1344), (1344, 320)])
def test_bf16_partial_last_round(lib, N, K):
    """4096 tokens with 1344 features make 96 tile pairs: more than one round of clusters,
    with a partial last round whose tiles the GEMM splits along the contraction (the
    parts' partial sums are added in a fixed order).  K = 320 leaves a half-filled last
    128-deep step; rows near the tile edges are always checked."""
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.choice(4096, 96, replace=False), [0, 255, 256, 3583, 3584, 4095]]))
    _run_case(4096, N, K, 16, 16.0, "bf16", seed=N + K, rows=rows)


def test_empty_batch(lib):
    q, _ = _quantized_weight(64, 128, 1)
    A = torch.randn(4, 128, device=DEV)
    B = torch.randn(64, 4, device=DEV)
    x = torch.empty(0, 128, device=DEV, dtype=torch.bfloat16)
    y, T = binding.qlora_linear_fwd(x, q, A, B, 8.0)
    assert y.shape == (0, 64)
    dy = torch.empty(0, 64, device=DEV, dtype=torch.bfloat16)
    dx, dA, dB = binding.qlora_linear_bwd(dy, x, T, q, A, B, 8.0,
                                          dA=torch.full((4, 128), 7.0, device=DEV),
                                          dB=torch.full((64, 4), 7.0, device=DEV))
    assert torch.all(dA == 0) and torch.all(dB == 0)


def test_shape_errors_are_explicit(lib):
    q, _ = _quantized_weight(64, 96, 1)
    x = torch.randn(4, 96, device=DEV, dtype=torch.bfloat16)
    with pytest.raises(binding.Nf4Error) as e:
        binding.qlora_linear_fwd(x, q, torch.randn(4, 96, device=DEV), torch.randn(64, 4, device=DEV), 8.0)
    assert e.value.status == binding.NF4_ERR_SHAPE


def test_linear_is_deterministic(lib):
    q, _ = _quantized_weight(520, 1024, 3)
    x = torch.randn(300, 1024, device=DEV, dtype=torch.bfloat16)
    dy = torch.randn(300, 520, device=DEV, dtype=torch.bfloat16)
    A = torch.randn(16, 1024, device=DEV) / 16
    B = torch.randn(520, 16, device=DEV) / 100
    outs = []
    for _ in range(2):
        y, T = binding.qlora_linear_fwd(x, q, A, B, 16.0)
        dx, dA, dB = binding.qlora_linear_bwd(dy, x, T, q, A, B, 16.0)
        outs.append([t.clone() for t in (y, T, dx, dA, dB)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("N,K", [(1344, 1344), (1024, 4096), (4096, 4096)])
def test_split_tiles_are_deterministic(lib, N, K):
    """4096 tokens: the GEMM's tile pairs leave a partial last round (1344 x 1344: 96 pairs,
    its 20 tail tiles cut into 3 equal parts each; 4096 x 4096: 256 pairs, 28 tail tiles in
    halves; 1024 x 4096: the forward's 64 pairs, fewer than the clusters, whole, and the
    dX's 256 in halves).  Whichever CTA finishes a split tile (the last part straight from
    its accumulator, or the last ticket from the parts' sums), the sum runs in the same
    order, so repeated calls give identical bits."""
    q, _ = _quantized_weight(N, K, 11)
    x = torch.randn(4096, K, device=DEV, dtype=torch.bfloat16)
    dy = torch.randn(4096, N, device=DEV, dtype=torch.bfloat16)
    A = torch.randn(16, K, device=DEV) / 16
    B = torch.randn(N, 16, device=DEV) / 100
    outs = []
    for _ in range(3):
        y, T = binding.qlora_linear_fwd(x, q, A, B, 16.0)
        dx, dA, dB = binding.qlora_linear_bwd(dy, x, T, q, A, B, 16.0)
        outs.append([t.clone() for t in (y, dx, dA, dB)])
    for later in outs[1:]:
        for a, b in zip(outs[0], later):
            assert torch.equal(a, b)


@pytest.mark.parametrize("M,N,K,r", [(64, 8, 64, 1), (130, 200, 192, 5), (300, 264, 576, 16),
                                     (511, 1032, 640, 64), (129, 136, 128, 128), (1, 520, 1024, 8),
                                     (5, 264, 576, 16), (16, 1032, 320, 64)])
def test_f16_profile_tiles_tails_and_small_m(lib, M, N, K, r):
    """The FP16 profile: IEEE half operands and outputs, fp32 accumulation, on the tiled path
    and (M <= 16) the small-M pass."""
    _run_case(M, N, K, r, 16.0, "f16", seed=N + 3)


def test_f16_profile_smollm2_qv_shapes(lib):
    c = wl.W2
    for name, N, K in c["shapes"]:
        if name in c["targets"]:
            _run_case(c["M"], N, K, c["r"], c["alpha"], "f16", seed=N + 5)


@pytest.mark.parametrize("name", ["gate_proj", "down_proj"])
def test_f16_profile_llama8b_sampled_rows(lib, name):
    c = wl.W3
    N, K = {n: (a, b) for n, a, b in c["shapes"]}[name]
    rows = np.sort(np.random.default_rng(6).choice(c["M"], 64, replace=False))
    _run_case(c["M"], N, K, c["r"], c["alpha"], "f16", seed=K + 1, dist="t", rows=rows)


def test_f16_profile_rslora_without_double_quant(lib):
    _run_case(96, 520, 512, 8, 16.0, "f16", mode=binding.SCALE_RSLORA, seed=3, dq=False)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,N,K,r", [(5, 40, 128, 3), (300, 264, 576, 16), (700, 1344, 1344, 16)])
def test_decoded_weight_entry_points_equal_the_nf4_calls(lib, dtype, M, N, K, r):
    """qlora_linear_fwd_w16 / _bwd_w16 with the weight as nf4_dequantize writes it: every output
    bit-identical to the tiled NF4-input calls (M > 16; at M <= 16 the NF4 forward takes the
    small-M pass, so the comparison there is the oracle's tolerance)."""
    q, w_deq = _quantized_weight(N, K, 31 + M)
    x = torch.from_numpy(wl.normal((M, K), 1.0, 1, 32 + M)).to(DEV).to(dtype)
    dy = torch.from_numpy(wl.normal((M, N), 1.0, 1, 33 + M)).to(DEV).to(dtype)
    A, B = (torch.from_numpy(t).to(DEV) for t in wl.adapters(N, K, r, 1, 34 + M))
    w16 = binding.nf4_dequantize(q, dtype)
    y, T = binding.qlora_linear_fwd(x, q, A, B, 16.0)
    y2, T2 = binding.qlora_linear_fwd_w16(x, w16, A, B, 16.0)
    dx, dA, dB = binding.qlora_linear_bwd(dy, x, T, q, A, B, 16.0)
    dx2, dA2, dB2 = binding.qlora_linear_bwd_w16(dy, x, T, w16, A, B, 16.0)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    same = [(dx, dx2), (dA, dA2), (dB, dB2)]
    if M > 16:
        same += [(y, y2), (T, T2)]
    for a, b in same:
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype != torch.float32 else b.view(torch.int32))
    if M <= 16:
        compute = "bf16" if dtype == torch.bfloat16 else "f16"
        xh = x.float().cpu().numpy()
        Ah, Bh = A.cpu().numpy(), B.cpu().numpy()
        s = qlora.lora_scale(16.0, r, "lora")
        y_ref, T_ref = qlora.forward(xh, w_deq, Ah, Bh, s, compute)
        fb = parity.forward_bounds(xh, w_deq, Ah, Bh, s, compute, y_ref, T_ref)
        parity.check({"y": y2.float().cpu().numpy(), "T": T2.cpu().numpy()}, {"y": y_ref, "T": T_ref},
                     {"y": fb["y"], "T": fb["T"]}, compute)


@pytest.mark.parametrize("compute", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K,r", [(17, 8, 64, 2), (65, 72, 128, 1), (511, 576, 576, 16), (1000, 192, 576, 17),
                                     (97, 1024, 1024, 32), (300, 520, 960, 24)])
def test_fused_small_shape_path(lib, compute, M, N, K, r):
    """Weights of at most 2^21 elements with K, N <= 1024 and rank <= 32 at M > 16 run the fused
    small-shape kernels (one forward launch, two backward): ragged token and feature tiles,
    ranks that fill 1 to 32 of the padded rank, the full-size limits."""
    _run_case(M, N, K, r, 16.0, compute, seed=M + N + r)


@pytest.mark.parametrize("M,N,K,r", [(130, 200, 192, 40), (300, 264, 576, 48)])
def test_tiled_path_small_ragged_shapes(lib, M, N, K, r):
    """A rank above 32 keeps small weights on the tiled tensor-core path: its ragged tiles at
    the shapes the fused path otherwise takes."""
    _run_case(M, N, K, r, 16.0, "bf16", seed=M + r)


def test_fused_small_shape_batch_forward_equals_single_calls(lib):
    """qlora_linear_fwd_batch runs its small-weight items in one fused launch (8 at most per
    launch) and the rest one call each; every item equals its single call bit for bit."""
    M = 384
    shapes = [(576, 576, 16), (192, 576, 16)] * 5 + [(1536, 576, 16)]
    items, singles = [], []
    for i, (N, K, r) in enumerate(shapes):
        q, _ = _quantized_weight(N, K, 70 + i)
        x = torch.from_numpy(wl.normal((M, K), 1.0, 1, 80 + i)).to(DEV).bfloat16()
        A, B = (torch.from_numpy(t).to(DEV) for t in wl.adapters(N, K, r, 1, 90 + i))
        items.append(dict(x=x, W=q, A=A, B=B, alpha=32.0))
        singles.append(binding.qlora_linear_fwd(x, q, A, B, 32.0))
    outs = binding.qlora_linear_fwd_batch(items)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    for (y, T), (y1, T1) in zip(outs, singles):
        assert torch.equal(y.view(torch.int16), y1.view(torch.int16))
        assert torch.equal(T.view(torch.int32), T1.view(torch.int32))


def test_batch_backward_equals_single_calls(lib):
    """qlora_linear_bwd_batch: the small-weight items (some with the stored weight, some with
    the decoded one) in fused groups of at most 8, the others one call each; every item equals
    its single qlora_linear_bwd bit for bit."""
    M = 300
    shapes = [(576, 576, 16), (192, 576, 16)] * 5 + [(1536, 576, 16), (264, 576, 5)]
    x = torch.from_numpy(wl.normal((M, 576), 1.0, 1, 111)).to(DEV).bfloat16()
    items, singles = [], []
    for i, (N, K, r) in enumerate(shapes):
        q, _ = _quantized_weight(N, K, 120 + i)
        A, B = (torch.from_numpy(t).to(DEV) for t in wl.adapters(N, K, r, 1, 130 + i))
        dy = torch.from_numpy(wl.normal((M, N), 1.0, 1, 140 + i)).to(DEV).bfloat16()
        _, T = binding.qlora_linear_fwd(x, q, A, B, 32.0)
        it = dict(dy=dy, x=x, T=T, A=A, B=B, alpha=32.0)
        if i % 3 == 1:
            it["w16"] = binding.nf4_dequantize(q, torch.bfloat16)
        else:
            it["W"] = q
        items.append(it)
        singles.append(binding.qlora_linear_bwd(dy, x, T, q, A, B, 32.0))
    outs = binding.qlora_linear_bwd_batch(items)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    for got, want in zip(outs, singles):
        assert torch.equal(got[0].view(torch.int16), want[0].view(torch.int16))
        assert torch.equal(got[1].view(torch.int32), want[1].view(torch.int32))
        assert torch.equal(got[2].view(torch.int32), want[2].view(torch.int32))
