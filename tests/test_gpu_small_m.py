"""Small-M forward parity on the Llama-3-8B-shaped matrices (the decode-like sweep).

Every one of the 7 projection matrices (q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096,
down 4096x14336) at M in {1, 2, 4, 8, 16} tokens, rank 8, alpha 16, with the LoRA scale
alpha/r and the rsLoRA scale alpha/sqrt(r), forward only; every output element is compared
with the float64 oracle (tests/parity.py criteria).  The stored NF4 bytes are seeded random
bytes (any byte pattern is a valid stored tensor), so the oracle decodes exactly what the
device reads without quantizing 218 M weights on the host; one matrix quantized by the oracle
from Student-t(5) weights keeps the realistic distribution in the set.
"""

import functools

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
C = wl.W4
SHAPES = {n: (N, K) for n, N, K in C["shapes"]}


def _to_device(ref, N, K):
    q = binding.Nf4Tensor.empty((N, K), ref["double_quant"], DEV)
    q.packed.copy_(torch.from_numpy(ref["packed"]))
    q.absmax.copy_(torch.from_numpy(np.asarray(ref["absmax"])))
    if ref["double_quant"]:
        q.nested_absmax.copy_(torch.from_numpy(ref["nested"]))
        q.offset[0] = float(ref["offset"])
    return q


def _decode_bf16_rows(ref, N, K):
    """The oracle's bf16 decode of an [N, K] NF4 tensor, in row chunks that hold whole nested
    groups (16384 elements), so no temporary is larger than about a million elements."""
    rows = 1
    while (rows * K) % (onf4.NESTED_BLOCK * onf4.BLOCK):
        rows += 1
    rows *= max(1, (1 << 20) // (rows * K))
    out = np.empty((N, K), dtype=np.float64)
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        e0, e1 = r0 * K, r1 * K
        b0, b1 = e0 // onf4.BLOCK, e1 // onf4.BLOCK
        g0, g1 = b0 // onf4.NESTED_BLOCK, -(-b1 // onf4.NESTED_BLOCK)
        part = dict(numel=e1 - e0, double_quant=True, packed=ref["packed"][e0 // 2:e1 // 2],
                    absmax=ref["absmax"][b0:b1], nested=ref["nested"][g0:g1], offset=ref["offset"])
        out[r0:r1] = onf4.dequantize(part, "bf16").reshape(r1 - r0, K)
    return out


@functools.lru_cache(maxsize=None)
def _stored(name):
    """(device NF4 tensor, the stored parts on the host) of one projection."""
    N, K = SHAPES[name]
    n = N * K
    if name == "k_proj":   # quantized by the oracle from Student-t(5) * 0.02 weights
        ref = onf4.quantize(wl.student_t((N, K), 5, 0.02, 4, 500), double_quant=True)
    else:
        parts = wl.random_nf4_parts((n + 1) // 2, onf4.num_blocks(n), onf4.num_nested(n), True, 4,
                                    600 + 10 * list(SHAPES).index(name))
        ref = dict(numel=n, double_quant=True, packed=parts["packed"], absmax=parts["absmax"],
                   nested=parts["nested"], offset=parts["offset"])
    return _to_device(ref, N, K), ref


@functools.lru_cache(maxsize=1)
def _matrix(name):
    """(device NF4 tensor, decoded weight rounded to bf16 as float64, its absolute values)."""
    N, K = SHAPES[name]
    q, ref = _stored(name)
    w64 = _decode_bf16_rows(ref, N, K)
    return q, w64, np.abs(w64)


def _inputs(name, M, N, K, r, seed):
    x = onf4.round_bf16(wl.normal((M, K), 1.0, 4, seed))
    A, B = wl.adapters(N, K, r, 4, seed + 1)
    return x, A, B


def _expect(x, w64, aw64, A, B, s):
    """Oracle y, T and their element-wise bounds on already rounded operands."""
    x64 = x.astype(np.float64)
    A64, B64 = (onf4.round_bf16(t).astype(np.float64) for t in (A, B))
    y, T = qlora.forward(x64, w64, A64, B64, s, compute="f64")
    b = parity.forward_bounds(x64, w64, A64, B64, s, "bf16", y, T, abs_W=aw64)
    return y, T, b


@pytest.mark.parametrize("name", list(SHAPES))
def test_small_m_forward_every_output(lib, name):
    N, K = SHAPES[name]
    q, w64, aw64 = _matrix(name)
    r, alpha = C["r"], C["alpha"]
    reports = {}
    for M in C["Ms"]:
        for mode, mname in ((binding.SCALE_LORA, "lora"), (binding.SCALE_RSLORA, "rslora")):
            x, A, B = _inputs(name, M, N, K, r, 10 * M + mode)
            s = qlora.lora_scale(alpha, r, mname)
            xd = torch.from_numpy(x).to(DEV).bfloat16()
            Ad, Bd = torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)
            y, T = binding.qlora_linear_fwd(xd, q, Ad, Bd, alpha, mode)
            torch.cuda.synchronize()
            y_ref, T_ref, b = _expect(x, w64, aw64, A, B, s)
            got = dict(y=y.float().cpu().numpy(), T=T.cpu().numpy())
            reports[(M, mname)] = parity.check(got, dict(y=y_ref, T=T_ref), b, "bf16")
    assert binding.device_status() == binding.NF4_OK
    worst = max(v["y"]["bound_ratio"] for v in reports.values())
    assert worst <= 1.0, reports


@pytest.mark.parametrize("M", [1, 16])
def test_small_m_layer_in_one_batch(lib, M):
    """The 7 projections of one layer through qlora_linear_fwd_batch (one T launch and one weight
    pass for all of them), each compared element by element with the oracle; a second call gives
    the same bits."""
    r, alpha = C["r"], C["alpha"]
    items, host = [], []
    for i, name in enumerate(SHAPES):
        N, K = SHAPES[name]
        q, _ = _stored(name)
        mode = binding.SCALE_RSLORA if i % 2 else binding.SCALE_LORA
        x, A, B = _inputs(name, M, N, K, r, 500 + 10 * i + M)
        items.append(dict(x=torch.from_numpy(x).to(DEV).bfloat16(), W=q, A=torch.from_numpy(A).to(DEV),
                          B=torch.from_numpy(B).to(DEV), alpha=alpha, mode=mode))
        host.append((name, x, A, B, qlora.lora_scale(alpha, r, "rslora" if mode else "lora")))
    outs = binding.qlora_linear_fwd_batch(items)
    first = [(y.clone(), T.clone()) for y, T in outs]
    again = binding.qlora_linear_fwd_batch(items)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    for (y0, T0), (y1, T1) in zip(first, again):
        assert torch.equal(y0, y1) and torch.equal(T0, T1)
    for (name, x, A, B, s), (y, T) in zip(host, first):
        _, w64, aw64 = _matrix(name)
        y_ref, T_ref, b = _expect(x, w64, aw64, A, B, s)
        parity.check(dict(y=y.float().cpu().numpy(), T=T.cpu().numpy()), dict(y=y_ref, T=T_ref), b, "bf16")


def _oracle_weight(N, K, seed, dq=True):
    ref = onf4.quantize(wl.normal((N, K), 0.02, 4, seed), double_quant=dq)
    q = _to_device(ref, N, K) if dq else None
    if not dq:
        q = binding.Nf4Tensor.empty((N, K), False, DEV)
        q.packed.copy_(torch.from_numpy(ref["packed"]))
        q.absmax.copy_(torch.from_numpy(ref["absmax"]))
    return q, onf4.round_bf16(onf4.dequantize(ref, "f32")).reshape(N, K).astype(np.float64)


@pytest.mark.parametrize("M", [1, 3, 8, 13, 16])
def test_small_m_ragged_shapes_and_ranks(lib, M):
    """Rows not a multiple of the 256-row tile, contractions not a multiple of the 256-deep span,
    ranks 1, 8, 64, 200 (one to four 64-wide slab boxes), double quantization on and off, in one
    batch and one by one."""
    cases = [(520, 576, 8, True), (264, 1088, 200, True), (8, 64, 1, True), (1032, 320, 64, False)]
    items, host = [], []
    for i, (N, K, r, dq) in enumerate(cases):
        q, w64 = _oracle_weight(N, K, 900 + i, dq)
        x, A, B = _inputs("ragged", M, N, K, r, 950 + 10 * i + M)
        mode = binding.SCALE_RSLORA if i == 1 else binding.SCALE_LORA
        items.append(dict(x=torch.from_numpy(x).to(DEV).bfloat16(), W=q, A=torch.from_numpy(A).to(DEV),
                          B=torch.from_numpy(B).to(DEV), alpha=16.0, mode=mode))
        host.append((x, w64, A, B, qlora.lora_scale(16.0, r, "rslora" if mode else "lora")))
    batched = binding.qlora_linear_fwd_batch(items)
    single = [binding.qlora_linear_fwd(it["x"], it["W"], it["A"], it["B"], it["alpha"], it["mode"]) for it in items]
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    for (x, w64, A, B, s), outs in zip(host, zip(batched, single)):
        y_ref, T_ref, b = _expect(x, w64, np.abs(w64), A, B, s)
        for y, T in outs:
            parity.check(dict(y=y.float().cpu().numpy(), T=T.cpu().numpy()), dict(y=y_ref, T=T_ref), b, "bf16")


def test_batch_refuses_a_bad_item(lib):
    q, _ = _oracle_weight(64, 128, 1)
    good = dict(x=torch.randn(4, 128, device=DEV).bfloat16(), W=q, A=torch.randn(4, 128, device=DEV),
                B=torch.randn(64, 4, device=DEV), alpha=8.0)
    bad = dict(good, A=torch.randn(4, 96, device=DEV))   # rank rows of the wrong length: W numel mismatch
    bad["W"] = _oracle_weight(64, 96, 2)[0]
    bad["x"] = torch.randn(4, 96, device=DEV).bfloat16()   # K = 96: not a multiple of 64
    with pytest.raises(binding.Nf4Error) as e:
        binding.qlora_linear_fwd_batch([good, bad])
    assert e.value.status == binding.NF4_ERR_SHAPE
