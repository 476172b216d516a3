"""Pins for the oracle's QLoRA linear forward and backward (CPU only).

The numpy float64 oracle is checked against pure-Python triple loops on tiny
shapes, against a finite-difference directional derivative of L = <y, R>, and
against closed forms (A = 0, B = 0, the two scale rules).
"""

import math

import numpy as np
import pytest

from oracle import nf4, qlora


def _tiny(seed, M=5, N=7, K=6, r=3):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((M, K)), rng.standard_normal((N, K)),
            rng.standard_normal((r, K)), rng.standard_normal((N, r)),
            rng.standard_normal((M, N)))


def _loops_forward(x, W, A, B, s):
    M, K = len(x), len(x[0])
    N, r = len(W), len(A)
    T = [[sum(x[m][k] * A[j][k] for k in range(K)) for j in range(r)] for m in range(M)]
    y = [[sum(x[m][k] * W[n][k] for k in range(K)) + s * sum(T[m][j] * B[n][j] for j in range(r))
          for n in range(N)] for m in range(M)]
    return np.array(y), np.array(T)


def _loops_backward(dy, x, W, A, B, s):
    M, K = len(x), len(x[0])
    N, r = len(W), len(A)
    T = [[sum(x[m][k] * A[j][k] for k in range(K)) for j in range(r)] for m in range(M)]
    G = [[sum(dy[m][n] * B[n][j] for n in range(N)) for j in range(r)] for m in range(M)]
    dX = [[sum(dy[m][n] * W[n][k] for n in range(N)) + s * sum(G[m][j] * A[j][k] for j in range(r))
           for k in range(K)] for m in range(M)]
    dA = [[s * sum(G[m][j] * x[m][k] for m in range(M)) for k in range(K)] for j in range(r)]
    dB = [[s * sum(dy[m][n] * T[m][j] for m in range(M)) for j in range(r)] for n in range(N)]
    return np.array(dX), np.array(dA), np.array(dB)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_backward_against_loops(seed):
    x, W, A, B, dy = _tiny(seed)
    s = 1.7
    y, T = qlora.forward(x, W, A, B, s, compute="f64")
    y2, T2 = _loops_forward(x.tolist(), W.tolist(), A.tolist(), B.tolist(), s)
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-12) and np.allclose(T, T2, rtol=1e-12, atol=1e-12)
    dX, dA, dB, _ = qlora.backward(dy, x, W, A, B, s, compute="f64")
    dX2, dA2, dB2 = _loops_backward(dy.tolist(), x.tolist(), W.tolist(), A.tolist(), B.tolist(), s)
    for got, want in ((dX, dX2), (dA, dA2), (dB, dB2)):
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_backward_is_the_gradient_of_forward():
    x, W, A, B, R = _tiny(4, M=4, N=5, K=6, r=2)
    s = 0.8
    dX, dA, dB, _ = qlora.backward(R, x, W, A, B, s, compute="f64")
    rng = np.random.default_rng(99)

    def loss(x_, A_, B_):
        return float(np.sum(qlora.forward(x_, W, A_, B_, s, compute="f64")[0] * R))

    eps = 1e-6
    for which, grad in (("x", dX), ("A", dA), ("B", dB)):
        d = rng.standard_normal(grad.shape)
        args_p = {"x": x, "A": A, "B": B}
        args_m = dict(args_p)
        args_p[which] = args_p[which] + eps * d
        args_m[which] = args_m[which] - eps * d
        fd = (loss(args_p["x"], args_p["A"], args_p["B"]) -
              loss(args_m["x"], args_m["A"], args_m["B"])) / (2 * eps)
        assert abs(fd - float(np.sum(grad * d))) <= 1e-6 * max(1.0, abs(fd))


def test_adapter_backward_matches_backward():
    x, W, A, B, dy = _tiny(12)
    dX, dA, dB, G = qlora.backward(dy, x, W, A, B, 1.3, compute="f64")
    dA2, dB2, G2 = qlora.adapter_backward(dy, x, A, B, 1.3, compute="f64")
    assert np.array_equal(dA, dA2) and np.array_equal(dB, dB2) and np.array_equal(G, G2)


def test_closed_forms():
    x, W, A, B, dy = _tiny(6)
    s = 2.0
    y, T = qlora.forward(x, W, np.zeros_like(A), B, s, compute="f64")
    assert np.allclose(y, x @ W.T) and np.all(T == 0)
    # B = 0 makes the adapter path vacuous: dA is structurally zero ([GATE] harness lesson)
    dX, dA, dB, G = qlora.backward(dy, x, W, A, np.zeros_like(B), s, compute="f64")
    assert np.all(dA == 0) and np.all(G == 0) and np.allclose(dX, dy @ W)
    assert not np.all(dB == 0)
    # doubling s doubles the adapter contributions only
    y1, _ = qlora.forward(x, W, A, B, 1.0, compute="f64")
    y2, _ = qlora.forward(x, W, A, B, 2.0, compute="f64")
    assert np.allclose(2 * (y1 - x @ W.T), y2 - x @ W.T)


def test_scale_rules_and_rank_bounds():
    assert qlora.lora_scale(16.0, 8, "lora") == 2.0
    assert qlora.lora_scale(32.0, 16, "lora") == 2.0
    assert qlora.lora_scale(16.0, 8, "rslora") == 16.0 / math.sqrt(8)
    assert qlora.lora_scale(1.0, 256) == 1.0 / 256
    for bad in (0, 257):
        with pytest.raises(ValueError):
            qlora.lora_scale(16.0, bad)


def test_bf16_profile_rounds_operands():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    W = rng.standard_normal((4, 64)).astype(np.float32)
    A = rng.standard_normal((2, 64)).astype(np.float32)
    B = rng.standard_normal((4, 2)).astype(np.float32)
    y, _ = qlora.forward(x, W, A, B, 1.0, compute="bf16")
    xr, Wr, Ar, Br = (nf4.round_bf16(t).astype(np.float64) for t in (x, W, A, B))
    assert np.allclose(y, xr @ Wr.T + (xr @ Ar.T) @ Br.T, rtol=1e-13, atol=1e-13)
    assert qlora.rel_frobenius(y, y) == 0.0
    assert qlora.linear_flops(2, 3, 4, 1) == 4 * 24 + 6 * 2 * 7
