"""Grouped calls on the tiled tensor-core path: consecutive items of qlora_linear_fwd_batch /
qlora_linear_bwd_batch that read the same x share one skinny pass over x (T in the forward,
dA in the backward), and a run's passes share launches.  With one input set every output
equals the single call's bit for bit; with several, dX and dB still do and y, T and dA agree
within the reordering of fp32 partial sums (each set's pass gets its share of the CTAs).  The
single calls are themselves checked against the oracle in tests/test_gpu_linear.py, so the
comparison carries that parity over to the runs.  The launch counts show that the grouping
happened.
"""

import pytest
import torch

from bit_nf4_quantized_gb300 import binding
from bit_nf4_quantized_gb300 import workloads as wl
from oracle import nf4 as onf4

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _weight(N, K, seed):
    ref = onf4.quantize(wl.normal((N, K), 0.02, 2, seed), double_quant=True)
    q = binding.Nf4Tensor.empty((N, K), True, DEV)
    q.packed.copy_(torch.from_numpy(ref["packed"]))
    q.absmax.copy_(torch.from_numpy(ref["absmax"]))
    q.nested_absmax.copy_(torch.from_numpy(ref["nested"]))
    q.offset[0] = float(ref["offset"])
    return q


def _same(a, b):
    if a.dtype in (torch.bfloat16, torch.float16):
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def _close(a, b, rtol):
    """fp32 tensors equal up to the order of their sums: within rtol of each element, or a
    tenth of that of the largest magnitude (a sum of K terms reordered moves by about K
    roundings of its partial sums, which near a zero result is large relative to it)."""
    return torch.allclose(a, b, rtol=rtol, atol=rtol * float(b.abs().max()) * 0.1)


def _single_set_runs(specs):
    """Per item: whether its run (up to 8 items in a row) holds one input set (items in a row
    on the same x whose ranks, each rounded up to 16, add up to at most 256)."""
    out = []
    for r0 in range(0, len(specs), 8):
        run = specs[r0:r0 + 8]
        sets, used, prev = 0, 0, None
        for N, K, r, alpha, mode, xid, decoded in run:
            nq = (r + 15) // 16 * 16
            if prev is None or xid != prev or used + nq > 256:
                sets, used = sets + 1, 0
            used += nq
            prev = xid
        out += [sets == 1] * len(run)
    return out


def _check_group(M, specs, seed, dtype=torch.bfloat16, device_weights=False):
    """specs: per item (N, K, r, alpha, mode, x_id, decoded).  Runs one forward batch and one
    backward batch over all items, and each item's single NF4-input calls; compares all.
    device_weights: the stored weights come from nf4_quantize on the device (large shapes;
    both sides read the same stored weight either way)."""
    xs = {}
    items_f, items_b, want_f, want_b, scales = [], [], [], [], []
    for i, (N, K, r, alpha, mode, xid, decoded) in enumerate(specs):
        if xid not in xs:
            xs[xid] = torch.from_numpy(wl.normal((M, K), 1.0, 1, seed + 500 + xid)).to(DEV).to(dtype)
        x = xs[xid]
        if device_weights:
            w = wl.device_student_t((N, K), 5, 0.02, seed + 10 * i, DEV, torch.bfloat16)
            q = binding.nf4_quantize(w, True)
        else:
            q = _weight(N, K, seed + 10 * i)
        A, B = (torch.from_numpy(t).to(DEV) for t in wl.adapters(N, K, r, 1, seed + 10 * i + 1))
        scales.append((B, alpha / r if mode == binding.SCALE_LORA else alpha / r ** 0.5))
        dy = torch.from_numpy(wl.normal((M, N), 1.0, 1, seed + 10 * i + 3)).to(DEV).to(dtype)
        y1, T1 = binding.qlora_linear_fwd(x, q, A, B, alpha, mode)
        want_f.append((y1, T1))
        want_b.append(binding.qlora_linear_bwd(dy, x, T1, q, A, B, alpha, mode))
        wsrc = dict(w16=binding.nf4_dequantize(q, dtype)) if decoded else dict(W=q)
        items_f.append(dict(x=x, A=A, B=B, alpha=alpha, mode=mode, **wsrc))
        items_b.append(dict(dy=dy, x=x, T=T1, A=A, B=B, alpha=alpha, mode=mode, **wsrc))
    torch.cuda.synchronize()
    n0 = binding.launch_count()
    got_f = binding.qlora_linear_fwd_batch(items_f)
    n1 = binding.launch_count()
    got_b = binding.qlora_linear_bwd_batch(items_b)
    n2 = binding.launch_count()
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    one_set = _single_set_runs(specs)
    for i, ((y, T), (y1, T1)) in enumerate(zip(got_f, want_f)):
        if one_set[i]:
            assert _same(y, y1), f"item {i}: y"
            assert _same(T, T1), f"item {i}: T"
        else:   # T's slices added in another order; y through a 16-bit s T
            assert _close(T, T1, 1e-4), f"item {i}: T"
            # each entry of the 16-bit s T may round one unit (2^-7 relative) the other way,
            # and y itself one unit
            B, sc = scales[i]
            bound = 2.0 ** -7 * (sc * (T1.abs() @ B.abs().T) + y1.float().abs()) + 1e-6
            assert torch.all((y.float() - y1.float()).abs() <= bound), f"item {i}: y"
    for i, (got, want) in enumerate(zip(got_b, want_b)):
        assert _same(got[0], want[0]), f"item {i}: dX"
        assert _same(got[2], want[2]), f"item {i}: dB"
        if one_set[i]:
            assert _same(got[1], want[1]), f"item {i}: dA"
        else:
            assert _close(got[1], want[1], 1e-4), f"item {i}: dA"
    return n1 - n0, n2 - n1


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_group_of_three_equals_single_calls(lib, dtype):
    """q, k, v-like items on one x with different ranks, scales and scale rules, weights given
    stored and decoded: one T pass and one dA pass for the three."""
    M, K = 300, 1280
    specs = [(1152, K, 16, 16.0, binding.SCALE_LORA, 0, True),
             (384, K, 8, 16.0, binding.SCALE_RSLORA, 0, False),
             (640, K, 24, 32.0, binding.SCALE_LORA, 0, True)]
    nf, nb = _check_group(M, specs, 7000, dtype)
    # forward: one batched decode (the stored weight), one staging, the T pass and its
    # finish, three GEMMs; backward: decode, staging, every G and dB pass in one launch and
    # their finishes in one more, three dX GEMMs, then the dA pass and its finish
    assert nf == 1 + 1 + 2 + 3
    assert nb == 1 + 1 + 2 + 3 + 2


def test_input_sets_break_at_x_changes_rank_and_count_limits(lib):
    """One run of items on x0, x0, x1, x0 (three input sets), ranks 128 + 128 + 16 (the third
    item opens a new set: at most 256 stacked rows) and nine items on one x (a run of 8, then
    the single call)."""
    M, K = 130, 1152
    specs = [(1104, K, 16, 16.0, binding.SCALE_LORA, 0, True), (1200, K, 16, 16.0, binding.SCALE_LORA, 0, True),
             (1048, K, 16, 16.0, binding.SCALE_LORA, 1, True), (1104, K, 16, 16.0, binding.SCALE_LORA, 0, True)]
    _check_group(M, specs, 7100)
    specs = [(1040, K, 128, 16.0, binding.SCALE_LORA, 0, True), (1088, K, 128, 16.0, binding.SCALE_LORA, 0, True),
             (1104, K, 16, 16.0, binding.SCALE_LORA, 0, False)]
    _check_group(M, specs, 7200)
    specs = [(1040 + 8 * i, K, 8, 16.0, binding.SCALE_LORA, 0, i % 2 == 0) for i in range(9)]
    _check_group(M, specs, 7300)


def test_llama8b_layer_run_equals_single_calls(lib):
    """The Llama-3-8B-shaped layer at 4096 tokens (r = 16, decoded weights) as the bench step
    runs it: q, k, v on one x, o on its own, gate and up on one x, down on its own."""
    M = 4096
    L = binding.SCALE_LORA
    specs = [(4096, 4096, 16, 16.0, L, 0, True), (1024, 4096, 16, 16.0, L, 0, True),
             (1024, 4096, 16, 16.0, L, 0, True), (4096, 4096, 16, 16.0, L, 1, True),
             (14336, 4096, 16, 16.0, L, 2, True), (14336, 4096, 16, 16.0, L, 2, True),
             (4096, 14336, 16, 16.0, L, 3, True)]
    nf, nb = _check_group(M, specs, 7400, device_weights=True)
    # forward: one staging launch (21 jobs), one T launch for the four input sets and its
    # finish, seven GEMMs; backward: one staging launch (32 jobs), one G/dB launch and its
    # finish, seven dX GEMMs, one dA launch and its finish
    assert nf == 1 + 2 + 7
    assert nb == 1 + 2 + 7 + 2


def test_small_m_batch_mixes_streamed_and_decoded_items(lib):
    """At M <= 16 the items given as NF4 go through the streaming pass (grouped) and the items
    given decoded through the tiled run (as qlora_linear_fwd_w16 does).  Decoded items equal
    their single calls bit for bit; streamed items differ from theirs only in the order of the
    fp32 partial sums (the group's split), so they agree within one bf16 rounding, plus the
    fp32 sums' own order error near zero."""
    M, K = 5, 1024
    x = torch.from_numpy(wl.normal((M, K), 1.0, 1, 7600)).to(DEV).bfloat16()
    specs = [(1152, 16, True), (384, 8, False), (640, 24, True), (1024, 16, False)]
    items, want, decoded = [], [], []
    for i, (N, r, dec) in enumerate(specs):
        q = _weight(N, K, 7610 + 10 * i)
        A, B = (torch.from_numpy(t).to(DEV) for t in wl.adapters(N, K, r, 1, 7611 + 10 * i))
        if dec:
            w16 = binding.nf4_dequantize(q, torch.bfloat16)
            want.append(binding.qlora_linear_fwd_w16(x, w16, A, B, 16.0))
            items.append(dict(x=x, w16=w16, A=A, B=B, alpha=16.0))
        else:
            want.append(binding.qlora_linear_fwd(x, q, A, B, 16.0))
            items.append(dict(x=x, W=q, A=A, B=B, alpha=16.0))
        decoded.append(dec)
    got = binding.qlora_linear_fwd_batch(items)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    for i, ((y, T), (y1, T1), dec) in enumerate(zip(got, want, decoded)):
        if dec:
            assert _same(y, y1), f"item {i}: y"
            assert _same(T, T1), f"item {i}: T"
        else:
            yf, y1f = y.float(), y1.float()
            assert torch.all((yf - y1f).abs() <= 2.0 ** -7 * y1f.abs() + 4e-6), f"item {i}: y"
            assert torch.allclose(T, T1, rtol=1e-5, atol=1e-6), f"item {i}: T"
