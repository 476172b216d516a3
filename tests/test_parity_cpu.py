"""CPU checks of the parity criteria in tests/parity.py.

A float32 emulation of the bf16 profile's arithmetic (operands rounded to bfloat16, float32
accumulation, bfloat16(s T) / bfloat16(s G) / bfloat16(G) / bfloat16(T) fed to the adapter
terms, bfloat16 outputs) must pass every criterion; the same emulation with a planted mistake
must fail: a dropped LoRA term, a slightly wrong 256 x 256 tile, a single wrong element.
"""

import numpy as np
import pytest

from oracle import nf4, qlora

import parity


def _case(seed, M=300, N=520, K=320, r=8):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    A = (rng.standard_normal((r, K)) / r).astype(np.float32)
    B = (rng.standard_normal((N, r)) * 0.01).astype(np.float32)
    dy = rng.standard_normal((M, N)).astype(np.float32)
    return x, W, A, B, dy


def _emulate(x, W, A, B, dy, s, drop_slab=False):
    """The device's bf16-profile arithmetic in float32 with its stated roundings."""
    b = nf4.round_bf16
    xb, Wb, Ab, Bb, dyb = (b(t) for t in (x, W, A, B, dy))
    T = xb @ Ab.T
    slab = b(np.float32(s) * T) @ Bb.T
    y = b(xb @ Wb.T + (0 if drop_slab else slab))
    G = dyb @ Bb
    dX = b(dyb @ Wb + b(np.float32(s) * G) @ Ab)
    dA = np.float32(s) * (b(G).T @ xb)
    dB = np.float32(s) * (dyb.T @ b(T))
    return dict(y=y, T=T, dX=dX, dA=dA, dB=dB)


def _check(got, x, W, A, B, dy, s):
    y, T = qlora.forward(x, W, A, B, s, "bf16")
    dX, dA, dB, _ = qlora.backward(dy, x, W, A, B, s, "bf16")
    fb = parity.forward_bounds(x, W, A, B, s, "bf16", y, T)
    bb = parity.backward_bounds(dy, x, W, A, B, s, "bf16", dX_ref=dX, dA_ref=dA, dB_ref=dB)
    want = dict(y=y, T=T, dX=dX, dA=dA, dB=dB)
    bounds = dict(y=fb["y"], T=fb["T"], **bb)
    return parity.check(got, want, bounds, "bf16")


@pytest.mark.parametrize("seed", [0, 1])
def test_emulated_device_arithmetic_passes(seed):
    x, W, A, B, dy = _case(seed)
    rep = _check(_emulate(x, W, A, B, dy, 2.0), x, W, A, B, dy, 2.0)
    assert rep["y"]["bound_ratio"] > 0.05     # the bound is not vacuous: rounding uses part of it


def test_dropped_lora_term_fails():
    x, W, A, B, dy = _case(2)
    with pytest.raises(AssertionError):
        _check(_emulate(x, W, A, B, dy, 2.0, drop_slab=True), x, W, A, B, dy, 2.0)


def test_one_slightly_wrong_tile_fails():
    x, W, A, B, dy = _case(3)
    got = _emulate(x, W, A, B, dy, 2.0)
    got["y"] = got["y"].copy()
    got["y"][256:, 256:512] *= np.float32(1.02)   # 2 % off on one block, 1/6 of the outputs
    with pytest.raises(AssertionError):
        _check(got, x, W, A, B, dy, 2.0)


def test_one_wrong_element_fails():
    x, W, A, B, dy = _case(4)
    got = _emulate(x, W, A, B, dy, 2.0)
    got["dX"] = got["dX"].copy()
    got["dX"][17, 33] = got["dX"][17, 33] * np.float32(1.03) + np.float32(1e-3)
    with pytest.raises(AssertionError):
        _check(got, x, W, A, B, dy, 2.0)
