"""Frozen-base QLoRA linear, forward and backward, in float64: plain CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages never typeset the formula; it follows from [ADAPT] section "One model
contract" (an NF4 base is frozen and needs an adapter), section "Packed NF4 and the
portable QLoRA profile" ("compute FP32 input gradients through the frozen base; no
base weight gradients are produced"), section "LoRA FA includes gradient
preconditioning" (s = alpha / rank) and section "Adapter API" (rank 1..256; rsLoRA
a separate method, whose primary paper fixes s = alpha / sqrt(rank)):

    T  = x A^T                       [M, r]   (kept for the backward pass)
    y  = x W^T + s T B^T             [M, N]
    G  = dY B                        [M, r]
    dX = dY W + s G A                [M, K]
    dA = s G^T x                     [r, K]
    dB = s dY^T T                    [N, r]

with W = deq(W_nf4) [N, K], A [r, K], B [N, r], no bias, no dropout.  [GATE] section
"The TFLOPS back-check" counts no dL/dW for the frozen base.

Precision: every product and sum here is float64 (numpy matmul is the library
step).  The operands are the exact values the device path multiplies: for the
bfloat16 profile x, dY, A, B and the decoded W are first rounded to bfloat16
(the decoded W as float32 nf4*a' then rounded once); for the half-precision
profile ([ADAPT] "Mixed precision keeps stable state in FP32": reconstructed
weights are rounded to FP16 before multiplication) the same operands are rounded
to IEEE binary16 instead; for the float32 profile they stay float32.  Results are compared with a relative Frobenius tolerance because
the accumulation order is not unique.
"""

import math

import numpy as np

from .nf4 import round_bf16, round_f16

RANK_MIN, RANK_MAX = 1, 256


def lora_scale(alpha: float, rank: int, mode: str = "lora") -> float:
    """s = alpha / rank (LoRA) or alpha / sqrt(rank) (rsLoRA); rank must be 1..256."""
    if not (RANK_MIN <= rank <= RANK_MAX):
        raise ValueError("rank out of range 1..256")
    if mode == "lora":
        return float(alpha) / rank
    if mode == "rslora":
        return float(alpha) / math.sqrt(rank)
    raise ValueError("unknown scale mode")


def _operands(compute: str, *arrays):
    """Operands as float64 after the rounding the device applies ('f64' keeps them unrounded)."""
    out = []
    for a in arrays:
        if compute == "f64":
            out.append(np.asarray(a, dtype=np.float64))
            continue
        a32 = np.asarray(a, dtype=np.float32)
        if compute == "bf16":
            a32 = round_bf16(a32)
        elif compute == "f16":
            a32 = round_f16(a32)
        elif compute != "f32":
            raise ValueError("compute must be 'bf16', 'f16', 'f32' or 'f64'")
        out.append(a32.astype(np.float64))
    return out


def forward(x, W, A, B, s: float, compute: str = "bf16"):
    """Return (y, T) in float64.  W is the decoded weight [N, K] (float32 values)."""
    x64, W64, A64, B64 = _operands(compute, x, W, A, B)
    T = x64 @ A64.T
    y = x64 @ W64.T + s * (T @ B64.T)
    return y, T


def backward(dy, x, W, A, B, s: float, compute: str = "bf16"):
    """Return (dX, dA, dB, G) in float64 for the loss gradient dy = dL/dy."""
    dy64, x64, W64, A64, B64 = _operands(compute, dy, x, W, A, B)
    T = x64 @ A64.T
    G = dy64 @ B64
    dX = dy64 @ W64 + s * (G @ A64)
    dA = s * (G.T @ x64)
    dB = s * (dy64.T @ T)
    return dX, dA, dB, G


def adapter_backward(dy, x, A, B, s: float, compute: str = "bf16"):
    """(dA, dB, G) alone -- the same formulas as ``backward`` without the M x N x K dX product."""
    dy64, x64, A64, B64 = _operands(compute, dy, x, A, B)
    T = x64 @ A64.T
    G = dy64 @ B64
    return s * (G.T @ x64), s * (dy64.T @ T), G


def forward_magnitudes(x, W, A, B, s: float, compute: str = "bf16", abs_W=None):
    """Sums of the absolute values of the terms of each output of ``forward``, in float64.

    Returns dict(y_base = |x| |W|^T (the terms x[m,k] W[n,k] of y), y_slab = |s| |T| |B|^T
    (the terms s T[m,j] B[n,j]), T = |x| |A|^T (the terms of T)), on the same rounded
    operands as ``forward``.  A rounding error of relative size u in every term of a sum
    moves that sum by at most u times these magnitudes, which is what element-wise error
    bounds are built from.  ``abs_W``: |W| of the rounded weight, when the caller already
    holds it (a large weight is then not converted again).
    """
    x64, A64, B64 = _operands(compute, x, A, B)
    aW = np.abs(_operands(compute, W)[0]) if abs_W is None else abs_W
    T_abs = np.abs(x64 @ A64.T)
    ax, aA, aB = (np.abs(t) for t in (x64, A64, B64))
    return dict(y_base=ax @ aW.T, y_slab=abs(s) * (T_abs @ aB.T), T=ax @ aA.T)


def backward_magnitudes(dy, x, W, A, B, s: float, compute: str = "bf16"):
    """Sums of |terms| of each output of ``backward`` (float64), as ``forward_magnitudes``:
    dX_base = |dY| |W|, dX_slab = |s| |G| |A|, G = |dY| |B|, dA = |s| |G|^T |x|,
    dB = |s| |dY|^T |T| with G = dY B and T = x A^T on the rounded operands.  With W = None
    the two dX entries are left out (the adapter gradients alone, no M x N x K product)."""
    dy64, x64, A64, B64 = _operands(compute, dy, x, A, B)
    G_abs = np.abs(dy64 @ B64)
    T_abs = np.abs(x64 @ A64.T)
    ady, ax, aA, aB = (np.abs(t) for t in (dy64, x64, A64, B64))
    out = dict(dX_slab=abs(s) * (G_abs @ aA), G=ady @ aB,
               dA=abs(s) * (G_abs.T @ ax), dB=abs(s) * (ady.T @ T_abs))
    if W is not None:
        out["dX_base"] = ady @ np.abs(_operands(compute, W)[0])
    return out


def rel_frobenius(got, want) -> float:
    """||got - want||_F / ||want||_F (0 when both are zero)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    num = np.linalg.norm(got - want)
    if den == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return float(num / den)


def tile_rel_frobenius(got, want, tile: int = 256) -> float:
    """Largest ``rel_frobenius`` over the tile x tile blocks of two 2-D arrays (ragged edge
    blocks included).  A block whose reference is all zero counts only if ``got`` differs."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    worst = 0.0
    for i in range(0, want.shape[0], tile):
        for j in range(0, want.shape[1], tile):
            worst = max(worst, rel_frobenius(got[i:i + tile, j:j + tile], want[i:i + tile, j:j + tile]))
    return worst


def linear_flops(M: int, N: int, K: int, r: int) -> int:
    """Algorithmic flops of one forward + backward: 4MNK base (y and dX) + 6Mr(N+K) adapter."""
    return 4 * M * N * K + 6 * M * r * (N + K)
