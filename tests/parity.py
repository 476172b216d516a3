"""Element-wise and tile-wise parity checks of the QLoRA linear against the float64 oracle.

The oracle runs on exactly the rounded operands the device multiplies (x, dY, A, B and the
decoded weight in bfloat16 for the bf16 profile), so what remains is the device's own
rounding, bounded element by element from the magnitudes of the terms of each sum
(``oracle.qlora.forward_magnitudes`` / ``backward_magnitudes``):

  u_out   the rounding of the output itself: 2^-8 relative for a bfloat16 output (half an ulp
          of an 8-bit significand), 2^-11 for IEEE half, 2^-24 for float32;
  u_op    the rounding of an intermediate that the profile feeds to a tensor-core slab or
          adapter pass: bfloat16(s T), bfloat16(s G), bfloat16(G), bfloat16(T) for the bf16
          profile (2^-8 of that intermediate's terms), float32 products for the fp32 profile;
  u_acc   float32 accumulation: for the tensor-core sums a fixed 2^-14 of the sum of |terms|
          (each 16-deep MMA step adds its products to a float32 accumulator; the measured
          errors sit far below this), for the fp32 profile the classic (n + 4) 2^-24 bound of
          a float32 sum of n terms in any order.

|got - want| <= u_out |want| + (1 + u_out) (u_acc mag + u_op mag_rounded + propagated error of
the intermediate) for every element, and the relative Frobenius error of every 256 x 256 block
stays <= 5e-3 (bf16) or 1e-5 (fp32), on top of the whole-array 2e-2 / 1e-5 of the stated
tolerance.  A whole or partly wrong tile, a missing split-K part or a missing LoRA term moves
its elements by far more than these bounds.
"""

import json
import os

import numpy as np

from oracle import qlora

FROB = {"f32": 1e-5, "bf16": 2e-2, "f16": 2e-2}
TILE_FROB = {"f32": 1e-5, "bf16": 5e-3, "f16": 5e-3}


def _units(compute, n_contract):
    if compute == "bf16":
        return dict(out=2.0 ** -8, op=2.0 ** -8, acc=2.0 ** -14)
    if compute == "f16":   # IEEE half: 11 significant bits, half an ulp is 2^-11 relative
        return dict(out=2.0 ** -11, op=2.0 ** -11, acc=2.0 ** -14)
    return dict(out=2.0 ** -24, op=2.0 ** -24, acc=(n_contract + 4) * 2.0 ** -24)


def forward_bounds(x, W, A, B, s, compute, y_ref, T_ref, abs_W=None):
    """Element-wise bounds for y and T of qlora_linear_fwd (``abs_W``: |W| if already held)."""
    K = np.shape(x)[1]
    r = np.shape(A)[0]
    u = _units(compute, K + r)
    fm = qlora.forward_magnitudes(x, W, A, B, s, compute, abs_W=abs_W)
    aB = np.abs(np.asarray(B, dtype=np.float64))
    t_err = u["acc"] * fm["T"]                          # error of the device's T itself
    y = u["out"] * np.abs(y_ref) + (1 + u["out"]) * (
        u["acc"] * (fm["y_base"] + fm["y_slab"]) + u["op"] * fm["y_slab"] + abs(s) * (t_err @ aB.T))
    T = 2.0 ** -24 * np.abs(T_ref) + t_err
    return dict(y=y, T=T)


def backward_bounds(dy, x, W, A, B, s, compute, dX_ref=None, dA_ref=None, dB_ref=None):
    """Element-wise bounds for dX (when W is given), dA and dB of qlora_linear_bwd."""
    N = np.shape(dy)[1]
    M, K = np.shape(x)
    r = np.shape(A)[0]
    u = _units(compute, N + r)
    bm = qlora.backward_magnitudes(dy, x, W, A, B, s, compute)
    fm_T = qlora.forward_magnitudes(x, np.zeros((1, K)), A, B, s, compute)["T"]
    aA = np.abs(np.asarray(A, dtype=np.float64))
    ax = np.abs(np.asarray(x, dtype=np.float64))
    ady = np.abs(np.asarray(dy, dtype=np.float64))
    g_err = u["acc"] * bm["G"]
    uM = _units(compute, M + r)["acc"]                  # dA and dB reduce over the tokens
    out = {}
    if W is not None:
        out["dX"] = u["out"] * np.abs(dX_ref) + (1 + u["out"]) * (
            u["acc"] * (bm["dX_base"] + bm["dX_slab"]) + u["op"] * bm["dX_slab"] + abs(s) * (g_err @ aA))
    if dA_ref is not None:
        out["dA"] = 2.0 ** -24 * np.abs(dA_ref) + (uM + u["op"]) * bm["dA"] + abs(s) * (g_err.T @ ax)
    if dB_ref is not None:
        out["dB"] = 2.0 ** -24 * np.abs(dB_ref) + (uM + u["op"]) * bm["dB"] + \
            abs(s) * (ady.T @ (u["acc"] * fm_T))
    return out


def check(got: dict, want: dict, bounds: dict, compute: str):
    """Assert the three criteria for every key of ``got``; returns the measured figures."""
    report = {}
    for k in got:
        g = np.asarray(got[k], dtype=np.float64)
        w = np.asarray(want[k], dtype=np.float64)
        b = np.asarray(bounds[k], dtype=np.float64) + 1e-35
        diff = np.abs(g - w)
        ratio = float(np.max(diff / b)) if diff.size else 0.0
        frob = qlora.rel_frobenius(g, w)
        tile = qlora.tile_rel_frobenius(g.reshape(g.shape[0], -1), w.reshape(w.shape[0], -1), 256)
        report[k] = dict(frob=frob, tile=tile, bound_ratio=ratio)
    if os.environ.get("PARITY_REPORT"):   # measured figures of every check, one JSON line each
        with open(os.environ["PARITY_REPORT"], "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "compute": compute, "report": report}) + "\n")
    for k, m in report.items():
        assert np.all(np.isfinite(np.asarray(got[k], dtype=np.float64))), (k, "non-finite", report)
        assert m["frob"] <= FROB[compute], (k, "relative Frobenius", report)
        assert m["tile"] <= TILE_FROB[compute], (k, "256 x 256 tile relative Frobenius", report)
        assert m["bound_ratio"] <= 1.0, (k, "element-wise bound", report)
    return report
