"""nf4_quantize_noalloc: quantization for callers that cannot allocate device memory.

A caller embedded in an engine that owns all device memory (or a loop where
cudaMalloc/cudaFree are not allowed) cannot hand nf4_quantize a workspace; this
entry point uses the library's own fixed scratch array instead.  These tests check,
through the C ABI, that it gives the same bytes as nf4_quantize on two calls in a
row (the second call must not be disturbed by what the first left in the shared
array), and that sizes above its limit are refused before any device work.

This file is named to be collected last.
"""

import ctypes

import pytest
import torch

from bit_nf4_quantized_gb300 import binding
from bit_nf4_quantized_gb300 import workloads as wl


def test_noalloc_refuses_sizes_above_the_limit():
    lib = binding.load()
    t = binding._Nf4Tensor()
    n = binding.NOALLOC_MAX_NUMEL + 1
    t.numel, t.double_quant, t.reserved = n, 1, 0
    t.packed, t.absmax, t.nested_absmax, t.offset = 0x10000000, 0x11000000, 0x12000000, 0x13000000
    x = ctypes.c_void_p(0x20000000)
    assert lib.nf4_quantize_noalloc(x, 0, n, ctypes.byref(t), None) == binding.NF4_ERR_TOO_LARGE
    assert lib.nf4_quantize_noalloc(None, 0, 100, ctypes.byref(t), None) == binding.NF4_ERR_ARG
    assert lib.nf4_quantize_noalloc(x, 0, 0, ctypes.byref(t), None) == binding.NF4_ERR_ARG


def _same(a, b):
    assert torch.equal(a.packed, b.packed)
    assert torch.equal(a.absmax, b.absmax)
    if a.double_quant:
        assert torch.equal(a.nested_absmax, b.nested_absmax)
        assert torch.equal(a.offset[:1], b.offset[:1])


@pytest.mark.gpu
def test_noalloc_matches_nf4_quantize_on_two_calls_in_a_row(lib):
    dev = "cuda"
    # first call: a large ragged fp32 tensor with outliers; second call: a smaller
    # bf16 tensor, so stale scratch from the first call would show if it were read
    first = torch.from_numpy(wl.with_outliers(wl.normal(64 * 256 * 37 + 29, 0.02, 5, 31), 0.001, 50.0, 5, 32))
    second = torch.from_numpy(wl.student_t(5000, 5, 0.02, 5, 33)).to(torch.bfloat16)
    for x in (first.to(dev), second.to(dev)):
        want = binding.nf4_quantize(x, double_quant=True)
        got = binding.nf4_quantize_noalloc(x, binding.Nf4Tensor.empty(tuple(x.shape), True, dev))
        torch.cuda.synchronize()
        _same(got, want)
    # without double quantization (fp32 block maxima; the scratch array is not used), twice
    for x in (second.to(dev), first.to(dev)):
        want = binding.nf4_quantize(x, double_quant=False)
        got = binding.nf4_quantize_noalloc(x, binding.Nf4Tensor.empty(tuple(x.shape), False, dev))
        torch.cuda.synchronize()
        _same(got, want)
    # the largest accepted size, then a small one again
    big = wl.device_normal((binding.NOALLOC_MAX_NUMEL,), 0.02, 91, dev, torch.bfloat16)
    _same(binding.nf4_quantize_noalloc(big, binding.Nf4Tensor.empty(tuple(big.shape), True, dev)),
          binding.nf4_quantize(big, double_quant=True))
    small = second.to(dev)
    _same(binding.nf4_quantize_noalloc(small, binding.Nf4Tensor.empty(tuple(small.shape), True, dev)),
          binding.nf4_quantize(small, double_quant=True))
    assert binding.device_status() == binding.NF4_OK
