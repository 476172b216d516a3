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


def test_rel_frobenius_hand_values():
    # got - want = [3, -1]: sqrt(10) over ||want|| = 5
    assert qlora.rel_frobenius([3.0, 4.0], [0.0, 5.0]) == math.sqrt(10.0) / 5.0
    # one wrong entry of a 2 x 2: |0.5| / sqrt(1 + 4 + 9 + 16)
    assert math.isclose(qlora.rel_frobenius([[1.0, 2.0], [3.0, 4.5]], [[1.0, 2.0], [3.0, 4.0]]),
                        0.5 / math.sqrt(30.0), rel_tol=1e-15)
    # not squared: scaling the error by 10 scales the result by 10
    assert math.isclose(qlora.rel_frobenius([0.0, 50.0], [0.0, 5.0]), 9.0, rel_tol=1e-15)
    assert qlora.rel_frobenius([0.0, 0.0], [0.0, 0.0]) == 0.0
    assert qlora.rel_frobenius([1e-30, 0.0], [0.0, 0.0]) == math.inf


def test_tile_rel_frobenius_finds_one_bad_tile():
    want = np.ones((512, 384))
    got = want.copy()
    got[256:, 256:] *= 1.1          # the ragged corner block (256 x 128) is 10 % off
    assert math.isclose(qlora.tile_rel_frobenius(got, want, 256), 0.1, rel_tol=1e-12)
    # the whole-array norm dilutes it: one block of 6 (1/6 of the entries)
    assert math.isclose(qlora.rel_frobenius(got, want), 0.1 * math.sqrt(256 * 128 / (512 * 384)), rel_tol=1e-12)
    assert qlora.tile_rel_frobenius(want, want) == 0.0


def _count_loop_flops(M, N, K, r):
    """Multiply-adds of the six products of one forward + backward, counted one by one in
    plain loops (T, x W^T, s T B^T, G, dY W, s G A, dA, dB); 2 flops each."""
    macs = 0
    for _m in range(M):                     # T = x A^T and y = x W^T + s T B^T
        for _j in range(r):
            macs += K
        for _n in range(N):
            macs += K + r
    for _m in range(M):                     # G = dY B and dX = dY W + s G A
        for _j in range(r):
            macs += N
        for _k in range(K):
            macs += N + r
    for _j in range(r):                     # dA = s G^T x
        for _k in range(K):
            macs += M
    for _n in range(N):                     # dB = s dY^T T
        for _j in range(r):
            macs += M
    return 2 * macs


def test_linear_flops_hand_count():
    for shape in ((2, 3, 4, 1), (3, 5, 7, 2), (4, 8, 6, 3)):
        assert qlora.linear_flops(*shape) == _count_loop_flops(*shape)
    # one Llama-3-8B-shaped projection (q_proj, 4096 x 4096) at 4096 tokens and rank 16, by hand:
    # 2 x 2 * 4096^3 for y and dX, plus 6 adapter products of 2 * 4096 * 4096 * 16 each
    assert qlora.linear_flops(4096, 4096, 4096, 16) == 274_877_906_944 + 6 * 536_870_912
    assert qlora.linear_flops(4096, 4096, 4096, 16) == 278_099_132_416


def test_magnitudes_hand_case():
    # x = [1, -2], W = [3, 4], A = [1, -1], B = [2], s = 0.5:
    # T = 1 + 2 = 3; y = 3 - 8 + 0.5 * 3 * 2 = -2; |terms| of y: 3 + 8 (base), 3 (slab)
    x, W, A, B = np.array([[1.0, -2.0]]), np.array([[3.0, 4.0]]), np.array([[1.0, -1.0]]), np.array([[2.0]])
    y, T = qlora.forward(x, W, A, B, 0.5, compute="f64")
    mag = qlora.forward_magnitudes(x, W, A, B, 0.5, compute="f64")
    assert y[0, 0] == -2.0 and T[0, 0] == 3.0
    assert mag["y_base"][0, 0] == 11.0 and mag["y_slab"][0, 0] == 3.0 and mag["T"][0, 0] == 3.0
    # backward with dY = [1]: G = 2; dX = [3, 4] + 0.5 * 2 * [1, -1] = [4, 3];
    # dA = 0.5 * 2 * [1, -2]; dB = 0.5 * 1 * 3
    dX, dA, dB, G = qlora.backward(np.array([[1.0]]), x, W, A, B, 0.5, compute="f64")
    bm = qlora.backward_magnitudes(np.array([[1.0]]), x, W, A, B, 0.5, compute="f64")
    assert dX.tolist() == [[4.0, 3.0]] and dA.tolist() == [[1.0, -2.0]] and dB.tolist() == [[1.5]]
    assert bm["dX_base"].tolist() == [[3.0, 4.0]] and bm["dX_slab"].tolist() == [[1.0, 1.0]]
    assert bm["dA"].tolist() == [[1.0, 2.0]] and bm["dB"].tolist() == [[1.5]] and bm["G"].tolist() == [[2.0]]


@pytest.mark.parametrize("seed", [3, 4])
def test_magnitudes_bound_and_equal_on_nonnegative_operands(seed):
    x, W, A, B, dy = _tiny(seed)
    s = 1.3
    # every term non-negative: the sums of |terms| are the outputs themselves
    ax, aW, aA, aB, ady = (np.abs(t) for t in (x, W, A, B, dy))
    y, T = qlora.forward(ax, aW, aA, aB, s, compute="f64")
    m = qlora.forward_magnitudes(ax, aW, aA, aB, s, compute="f64")
    assert np.allclose(m["y_base"] + m["y_slab"], y, rtol=1e-14) and np.allclose(m["T"], T, rtol=1e-14)
    dX, dA, dB, G = qlora.backward(ady, ax, aW, aA, aB, s, compute="f64")
    bm = qlora.backward_magnitudes(ady, ax, aW, aA, aB, s, compute="f64")
    for got, want in ((bm["dX_base"] + bm["dX_slab"], dX), (bm["dA"], dA), (bm["dB"], dB), (bm["G"], G)):
        assert np.allclose(got, want, rtol=1e-14)
    # signed operands: each output is bounded by its magnitude (triangle inequality)
    y, T = qlora.forward(x, W, A, B, -s, compute="f64")
    m = qlora.forward_magnitudes(x, W, A, B, -s, compute="f64")
    assert np.all(np.abs(y) <= m["y_base"] + m["y_slab"] + 1e-12) and np.all(np.abs(T) <= m["T"] + 1e-12)
    dX, dA, dB, G = qlora.backward(dy, x, W, A, B, -s, compute="f64")
    bm = qlora.backward_magnitudes(dy, x, W, A, B, -s, compute="f64")
    assert np.all(np.abs(dX) <= bm["dX_base"] + bm["dX_slab"] + 1e-12)
    assert np.all(np.abs(dA) <= bm["dA"] + 1e-12) and np.all(np.abs(dB) <= bm["dB"] + 1e-12)


def test_f16_profile_rounds_operands():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    W = (rng.standard_normal((4, 64)) * 0.02).astype(np.float32)
    A = rng.standard_normal((2, 64)).astype(np.float32)
    B = rng.standard_normal((4, 2)).astype(np.float32)
    y, T = qlora.forward(x, W, A, B, 1.5, compute="f16")
    xr, Wr, Ar, Br = (nf4.round_f16(t).astype(np.float64) for t in (x, W, A, B))
    assert np.allclose(y, xr @ Wr.T + 1.5 * (xr @ Ar.T) @ Br.T, rtol=1e-13, atol=1e-13)
    # the operands really were rounded: the result differs from the bf16 and fp32 profiles
    assert not np.allclose(y, qlora.forward(x, W, A, B, 1.5, compute="bf16")[0], rtol=1e-6, atol=0)
    assert not np.allclose(y, qlora.forward(x, W, A, B, 1.5, compute="f32")[0], rtol=1e-9, atol=0)
