"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, its size queries and tables agree with the oracle, and invalid
arguments are refused before any device work (no compute call is made here)."""

import ctypes
import os
import re

import numpy as np
import pytest

from bit_nf4_quantized_gb300 import binding, build
from oracle import codebooks as cb
from oracle import nf4 as onf4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.append(m.group(1))
    return sorted(set(names))


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding.ENTRY_POINTS) <= set(names)
    assert lib.nf4_abi_version() == 5


def test_noalloc_limit_has_one_source(lib):
    """The binding's NOALLOC_MAX_NUMEL is the header's NF4_QUANTIZE_NOALLOC_MAX_NUMEL, and the
    library refuses exactly the sizes above it (a refusal comes before any device work)."""
    text = open(os.path.join(ROOT, "include", "qlora_nf4.h")).read()
    m = re.search(r"#define\s+NF4_QUANTIZE_NOALLOC_MAX_NUMEL\s+\((\d+)LL\)", text)
    assert m and int(m.group(1)) == binding.NOALLOC_MAX_NUMEL
    t = binding._Nf4Tensor()
    n = binding.NOALLOC_MAX_NUMEL + 1
    t.numel, t.double_quant, t.reserved = n, 0, 0
    t.packed, t.absmax = 0x10000000, 0x11000000
    assert lib.nf4_quantize_noalloc(ctypes.c_void_p(0x20000000), 0, n, ctypes.byref(t), None) == \
        binding.NF4_ERR_TOO_LARGE


def test_size_queries_match_oracle(lib):
    for n in (1, 2, 63, 64, 65, 16383, 16384, 16385, 576 * 576, 4096 * 14336, 2 ** 30, 2 ** 31 + 5):
        assert lib.nf4_num_blocks(n) == onf4.num_blocks(n)
        assert lib.nf4_num_nested(n) == onf4.num_nested(n)
        assert lib.nf4_packed_bytes(n, 1) == onf4.packed_bytes(n, True)
        assert lib.nf4_packed_bytes(n, 0) == onf4.packed_bytes(n, False)
    assert lib.nf4_packed_bytes(0, 1) == 0


def test_tables_equal_oracle_bit_for_bit():
    nf4, dyn8 = binding.code_tables()
    assert np.array_equal(np.array(nf4, np.float32).view(np.uint32), cb.nf4_codebook().view(np.uint32))
    assert np.array_equal(np.array(dyn8, np.float32).view(np.uint32),
                          cb.dynamic8_codebook().view(np.uint32))


def _fake_tensor(numel, dq=1, base=0x10000000):
    t = binding._Nf4Tensor()
    t.numel, t.double_quant, t.reserved = numel, dq, 0
    t.packed, t.absmax = base, base + 0x100000
    t.nested_absmax = base + 0x200000 if dq else None
    t.offset = base + 0x300000 if dq else None
    return t


def test_validation_refuses_bad_arguments(lib):
    x = ctypes.c_void_p(0x20000000)
    ws = ctypes.c_void_p(0x30000000)
    t = _fake_tensor(1000)
    q = lambda *a: lib.nf4_quantize(*a)  # noqa: E731
    assert q(None, 0, 1000, ctypes.byref(t), ws, 1 << 20, None) == binding.NF4_ERR_ARG
    assert q(x, 0, 0, ctypes.byref(t), ws, 1 << 20, None) == binding.NF4_ERR_ARG
    assert q(x, 7, 1000, ctypes.byref(t), ws, 1 << 20, None) == binding.NF4_ERR_DTYPE
    assert q(x, 0, 999, ctypes.byref(t), ws, 1 << 20, None) == binding.NF4_ERR_CORRUPT
    assert q(ctypes.c_void_p(0x20000004), 0, 1000, ctypes.byref(t), ws, 1 << 20, None) == binding.NF4_ERR_ALIGN
    assert q(x, 0, 1000, ctypes.byref(t), ws, 8, None) == binding.NF4_ERR_WORKSPACE
    bad = _fake_tensor(1000)
    bad.nested_absmax = None
    assert q(x, 0, 1000, ctypes.byref(bad), ws, 1 << 20, None) == binding.NF4_ERR_CORRUPT
    nodq = _fake_tensor(1000, dq=0)
    nodq.offset = 0x40000000
    assert q(x, 0, 1000, ctypes.byref(nodq), ws, 1 << 20, None) == binding.NF4_ERR_CORRUPT

    # the batch: every item checked before anything is enqueued
    items = (binding._QuantItem * 2)()
    items[0] = binding._QuantItem(x.value, 0, 1000, ctypes.pointer(t))
    items[1] = binding._QuantItem(x.value, 1, 1000, ctypes.pointer(t))
    qb = lambda n, wsz=1 << 20, w=ws: lib.nf4_quantize_batch(n, items, w, wsz, None)  # noqa: E731
    assert qb(0) == binding.NF4_ERR_ARG
    assert qb(2, wsz=8) == binding.NF4_ERR_WORKSPACE
    assert lib.nf4_quantize_batch_workspace_bytes(2, items) == 2 * lib.nf4_quantize_workspace_bytes(1000, 1)
    items[1] = binding._QuantItem(x.value, binding.NF4_F16, 1000, ctypes.pointer(t))
    assert qb(2) == binding.NF4_ERR_DTYPE
    items[1] = binding._QuantItem(0x20000004, 1, 1000, ctypes.pointer(t))
    assert qb(2) == binding.NF4_ERR_ALIGN
    items[1] = binding._QuantItem(x.value, 1, 999, ctypes.pointer(t))
    assert qb(2) == binding.NF4_ERR_CORRUPT

    assert lib.nf4_dequantize(None, x, 0, None) == binding.NF4_ERR_ARG
    assert lib.nf4_dequantize(ctypes.byref(t), x, 3, None) == binding.NF4_ERR_DTYPE
    # half precision: an output of the dequantize and a compute dtype of the linear, not an
    # input of the quantizer nor an output of the selected-row and merge calls
    assert q(x, binding.NF4_F16, 1000, ctypes.byref(t), ws, 1 << 20, None) == binding.NF4_ERR_DTYPE

    w = _fake_tensor(64 * 128)
    p = ctypes.c_void_p(0x50000000)
    f = lambda M, N, K, r, alpha=16.0, mode=0, cd=1, wt=w, wsz=1 << 30: lib.qlora_linear_fwd(  # noqa: E731
        M, N, K, r, ctypes.c_float(alpha), mode, cd, p, ctypes.byref(wt), p, p, p, p, ws, wsz, None)
    assert f(4, 64, 128, 0) == binding.NF4_ERR_ARG            # rank below 1
    assert f(4, 64, 128, 257) == binding.NF4_ERR_ARG          # rank above 256
    assert f(4, 64, 128, 65) == binding.NF4_ERR_ARG           # rank above min(N, K)
    assert f(4, 64, 128, 8, alpha=float("nan")) == binding.NF4_ERR_ARG
    assert f(4, 64, 128, 8, mode=5) == binding.NF4_ERR_ARG
    assert f(4, 64, 128, 8, cd=9) == binding.NF4_ERR_DTYPE
    w2 = _fake_tensor(100 * 96)
    assert f(4, 100, 96, 8, wt=w2) == binding.NF4_ERR_SHAPE  # bf16 needs K % 64 == 0
    assert f(4, 100, 96, 8, cd=binding.NF4_F16, wt=w2) == binding.NF4_ERR_SHAPE   # and so does half
    w3 = _fake_tensor(100 * 128)
    assert f(4, 100, 128, 8, wt=w3) == binding.NF4_ERR_SHAPE  # bf16 needs N % 8 == 0
    assert f(4, 64, 64, 8) == binding.NF4_ERR_CORRUPT        # numel != N*K
    if lib.qlora_fwd_workspace_bytes(4, 64, 128, 8, 1) > 0:
        assert f(4, 64, 128, 8, wsz=1) == binding.NF4_ERR_WORKSPACE
    b = lambda wsz: lib.qlora_linear_bwd(  # noqa: E731
        4, 64, 128, 8, ctypes.c_float(16.0), 0, 1, p, p, p, ctypes.byref(w), p, p, p, p, p, ws, wsz, None)
    assert b(0) == binding.NF4_ERR_WORKSPACE

    # the decoded-weight entry points: 16-bit compute only, a 16-byte aligned weight
    fw = lambda M, N, K, r, cd=1, w16=p, wsz=1 << 30: lib.qlora_linear_fwd_w16(  # noqa: E731
        M, N, K, r, ctypes.c_float(16.0), 0, cd, p, w16, p, p, p, p, ws, wsz, None)
    assert fw(4, 64, 128, 8, cd=binding.NF4_F32) == binding.NF4_ERR_DTYPE
    assert fw(4, 64, 128, 8, w16=None) == binding.NF4_ERR_ARG
    assert fw(4, 64, 128, 8, w16=ctypes.c_void_p(0x50000002)) == binding.NF4_ERR_ALIGN
    assert fw(4, 100, 96, 8) == binding.NF4_ERR_SHAPE
    assert fw(4, 64, 128, 8, wsz=1) == binding.NF4_ERR_WORKSPACE
    assert lib.qlora_fwd_w16_workspace_bytes(4, 64, 128, 8, binding.NF4_F32) == 0
    assert 0 < lib.qlora_fwd_w16_workspace_bytes(4096, 14336, 4096, 16, 1) < lib.qlora_fwd_workspace_bytes(
        4096, 14336, 4096, 16, 1)
    bw = lambda cd=1, w16=p, wsz=1 << 30: lib.qlora_linear_bwd_w16(  # noqa: E731
        4, 64, 128, 8, ctypes.c_float(16.0), 0, cd, p, p, p, w16, p, p, p, p, p, ws, wsz, None)
    assert bw(cd=binding.NF4_F32) == binding.NF4_ERR_DTYPE
    assert bw(w16=None) == binding.NF4_ERR_ARG
    assert bw(wsz=1) == binding.NF4_ERR_WORKSPACE

    # selected embedding rows: E [100, 64]
    e = _fake_tensor(100 * 64)
    emb = lambda rows, dim, ids, n, out, od=0, et=e: lib.nf4_embedding_rows(  # noqa: E731
        ctypes.byref(et) if et is not None else None, rows, dim, ids, n, out, od, None)
    assert emb(100, 64, p, 4, p, et=None) == binding.NF4_ERR_ARG
    assert emb(0, 64, p, 4, p) == binding.NF4_ERR_ARG
    assert emb(100, 64, p, -1, p) == binding.NF4_ERR_ARG
    assert emb(100, 64, p, 4, p, od=4) == binding.NF4_ERR_DTYPE
    assert emb(100, 64, p, 4, p, od=binding.NF4_F16) == binding.NF4_ERR_DTYPE
    assert emb(100, 32, p, 4, p) == binding.NF4_ERR_CORRUPT          # numel != rows*dim
    assert emb(100, 64, None, 0, None) == binding.NF4_OK             # no ids: nothing to do
    assert emb(100, 64, None, 4, p) == binding.NF4_ERR_ARG
    assert emb(100, 64, p, 4, ctypes.c_void_p(0x50000008)) == binding.NF4_ERR_ALIGN

    # merged weight: W [64, 128]
    m = lambda N, K, r, od=0, wt=w, a=p, alpha=16.0, mode=0: lib.nf4_merge_lora(  # noqa: E731
        N, K, r, ctypes.c_float(alpha), mode, ctypes.byref(wt), a, p, p, od, None)
    assert m(64, 128, 8, od=binding.NF4_F16) == binding.NF4_ERR_DTYPE
    assert m(64, 128, 8, od=3) == binding.NF4_ERR_DTYPE
    assert m(64, 128, 0) == binding.NF4_ERR_ARG
    assert m(64, 128, 65) == binding.NF4_ERR_ARG
    assert m(64, 128, 8, alpha=float("inf")) == binding.NF4_ERR_ARG
    assert m(64, 128, 8, mode=3) == binding.NF4_ERR_ARG
    assert m(64, 124, 8, wt=_fake_tensor(64 * 124)) == binding.NF4_ERR_SHAPE   # K % 8
    assert m(64, 64, 8) == binding.NF4_ERR_CORRUPT                             # numel != N*K
    assert m(64, 128, 8, a=ctypes.c_void_p(0x50000004)) == binding.NF4_ERR_ALIGN
    assert m(64, 128, 8, a=None) == binding.NF4_ERR_ARG


def test_dequantize_batch_validation(lib):
    """nf4_dequantize_batch checks every item before enqueueing anything (no device work)."""
    t = _fake_tensor(1000)
    items = (binding._DequantItem * 2)()
    items[0].w = ctypes.pointer(t)
    items[0].y = 0x50000000
    items[1].w = ctypes.pointer(t)
    items[1].y = None
    bf16 = binding.NF4_BF16
    assert lib.nf4_dequantize_batch(0, items, bf16, None) == binding.NF4_ERR_ARG
    assert lib.nf4_dequantize_batch(1, None, bf16, None) == binding.NF4_ERR_ARG
    assert lib.nf4_dequantize_batch(1, items, 9, None) == binding.NF4_ERR_DTYPE
    assert lib.nf4_dequantize_batch(2, items, bf16, None) == binding.NF4_ERR_ARG     # item 1: no output
    items[1].y = 0x50000008
    assert lib.nf4_dequantize_batch(2, items, bf16, None) == binding.NF4_ERR_ALIGN   # item 1: misaligned
    bad = _fake_tensor(1000)
    bad.nested_absmax = None
    items[1].w = ctypes.pointer(bad)
    items[1].y = 0x50001000
    assert lib.nf4_dequantize_batch(2, items, bf16, None) != binding.NF4_OK          # item 1: no nested maxima


def test_status_strings(lib):
    for s in range(10):
        assert lib.nf4_status_str(s).decode()
    assert lib.nf4_status_str(99).decode() == "unknown status"


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        binding.load()


def test_group_workspace_covers_each_single_layout(lib):
    """The batch workspace of a run of tiled items holds every item's single-call workspace,
    whether the items share x or not, plus the shared passes' buffers."""
    M, r = 1000, 16
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096)]
    single = [lib.qlora_fwd_w16_workspace_bytes(M, N, K, r, 1) for N, K in shapes]
    grouped = binding.qlora_fwd_batch_workspace_bytes(M, shapes, r, xs=[0, 0, 0], w16=True)
    apart = binding.qlora_fwd_batch_workspace_bytes(M, shapes, r, xs=[0, 1, 2], w16=True)
    assert grouped >= sum(single)
    assert apart >= sum(single)
    single_b = [lib.qlora_bwd_w16_workspace_bytes(M, N, K, r, 1) for N, K in shapes]
    grouped_b = binding.qlora_bwd_batch_workspace_bytes(M, shapes, r, xs=[0, 0, 0], w16=True)
    apart_b = binding.qlora_bwd_batch_workspace_bytes(M, shapes, r, xs=[0, 1, 2], w16=True)
    assert grouped_b >= sum(single_b)
    assert apart_b >= sum(single_b)
    # a group of one is the single call; nine items on one x run as 8 + 1
    assert binding.qlora_fwd_batch_workspace_bytes(M, shapes[:1], r, w16=True) == single[0]
    nine = binding.qlora_fwd_batch_workspace_bytes(M, [(1024, 4096)] * 9, r, xs=[0] * 9, w16=True)
    eight = binding.qlora_fwd_batch_workspace_bytes(M, [(1024, 4096)] * 8, r, xs=[0] * 8, w16=True)
    assert nine == eight
