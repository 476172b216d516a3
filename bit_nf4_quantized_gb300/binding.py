"""Thin Python binding of libqlora_nf4.so (ctypes): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module only
allocates outputs and workspaces with PyTorch, passes device pointers and the
current CUDA stream through the C ABI declared in ``include/qlora_nf4.h``, and turns
a non-OK status into :class:`Nf4Error`.  There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

NF4_OK, NF4_ERR_ARG, NF4_ERR_SHAPE, NF4_ERR_ALIGN, NF4_ERR_DTYPE = 0, 1, 2, 3, 4
NF4_ERR_NONFINITE, NF4_ERR_CORRUPT, NF4_ERR_CUDA, NF4_ERR_TIMEOUT, NF4_ERR_WORKSPACE = 5, 6, 7, 8, 9
NF4_ERR_TOO_LARGE = 10
NOALLOC_MAX_NUMEL = 1 << 26
NF4_F32, NF4_BF16, NF4_F16 = 0, 1, 2
SCALE_LORA, SCALE_RSLORA = 0, 1

ENTRY_POINTS = (
    "nf4_abi_version", "nf4_status_str", "nf4_num_blocks", "nf4_num_nested", "nf4_packed_bytes",
    "nf4_code_tables", "nf4_quantize_workspace_bytes", "nf4_quantize", "nf4_dequantize",
    "nf4_embedding_rows", "nf4_merge_lora",
    "qlora_fwd_workspace_bytes", "qlora_bwd_workspace_bytes", "qlora_linear_fwd",
    "qlora_linear_bwd", "qlora_last_device_status", "nf4_kernel_launch_count",
    "qlora_fwd_batch_workspace_bytes", "qlora_linear_fwd_batch",
    "qlora_fwd_w16_workspace_bytes", "qlora_bwd_w16_workspace_bytes", "qlora_linear_fwd_w16",
    "qlora_linear_bwd_w16", "nf4_quantize_batch_workspace_bytes", "nf4_quantize_batch",
    "qlora_bwd_batch_workspace_bytes", "qlora_linear_bwd_batch", "nf4_dequantize_batch",
)


class Nf4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_status_str(status)} (status {status})")


class _Nf4Tensor(ctypes.Structure):
    _fields_ = [("numel", ctypes.c_int64), ("double_quant", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("packed", ctypes.c_void_p),
                ("absmax", ctypes.c_void_p), ("nested_absmax", ctypes.c_void_p),
                ("offset", ctypes.c_void_p)]


class _FwdItem(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("rank", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("mode", ctypes.c_int32), ("W", ctypes.POINTER(_Nf4Tensor)),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("T_out", ctypes.c_void_p), ("w16", ctypes.c_void_p)]


class _BwdItem(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("rank", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("mode", ctypes.c_int32), ("W", ctypes.POINTER(_Nf4Tensor)),
                ("w16", ctypes.c_void_p), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("dy", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("T", ctypes.c_void_p), ("dx", ctypes.c_void_p), ("dA", ctypes.c_void_p),
                ("dB", ctypes.c_void_p)]


class _QuantItem(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_dtype", ctypes.c_int32), ("numel", ctypes.c_int64),
                ("out", ctypes.POINTER(_Nf4Tensor))]


class _DequantItem(ctypes.Structure):
    _fields_ = [("w", ctypes.POINTER(_Nf4Tensor)), ("y", ctypes.c_void_p)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the in-tree library (build it first with ``bit_nf4_quantized_gb300.build``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libqlora_nf4.so is not built ({path}); run bit_nf4_quantized_gb300.build")
    lib = ctypes.CDLL(path)
    i64, i32, sz, vp, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
    tp = ctypes.POINTER(_Nf4Tensor)
    sig = {
        "nf4_abi_version": (i32, []),
        "nf4_status_str": (ctypes.c_char_p, [i32]),
        "nf4_num_blocks": (i64, [i64]),
        "nf4_num_nested": (i64, [i64]),
        "nf4_packed_bytes": (sz, [i64, i32]),
        "nf4_code_tables": (None, [vp, vp]),
        "nf4_quantize_workspace_bytes": (sz, [i64, i32]),
        "nf4_quantize": (i32, [vp, i32, i64, tp, vp, sz, vp]),
        "nf4_dequantize": (i32, [tp, vp, i32, vp]),
        "nf4_quantize_batch_workspace_bytes": (sz, [i32, ctypes.POINTER(_QuantItem)]),
        "nf4_quantize_batch": (i32, [i32, ctypes.POINTER(_QuantItem), vp, sz, vp]),
        "nf4_quantize_noalloc": (i32, [vp, i32, i64, tp, vp]),
        "nf4_dequantize_batch": (i32, [i32, ctypes.POINTER(_DequantItem), i32, vp]),
        "nf4_embedding_rows": (i32, [tp, i64, i64, vp, i64, vp, i32, vp]),
        "nf4_merge_lora": (i32, [i64, i64, i32, f32, i32, tp, vp, vp, vp, i32, vp]),
        "qlora_fwd_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "qlora_bwd_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "qlora_linear_fwd": (i32, [i64, i64, i64, i32, f32, i32, i32, vp, tp, vp, vp, vp, vp, vp, sz, vp]),
        "qlora_linear_bwd": (i32, [i64, i64, i64, i32, f32, i32, i32, vp, vp, vp, tp, vp, vp,
                                   vp, vp, vp, vp, sz, vp]),
        "qlora_fwd_batch_workspace_bytes": (sz, [i64, i32, ctypes.POINTER(_FwdItem), i32]),
        "qlora_linear_fwd_batch": (i32, [i64, i32, ctypes.POINTER(_FwdItem), i32, vp, sz, vp]),
        "qlora_fwd_w16_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "qlora_bwd_w16_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "qlora_linear_fwd_w16": (i32, [i64, i64, i64, i32, f32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "qlora_linear_bwd_w16": (i32, [i64, i64, i64, i32, f32, i32, i32, vp, vp, vp, vp, vp, vp,
                                       vp, vp, vp, vp, sz, vp]),
        "qlora_bwd_batch_workspace_bytes": (sz, [i64, i32, ctypes.POINTER(_BwdItem), i32]),
        "qlora_linear_bwd_batch": (i32, [i64, i32, ctypes.POINTER(_BwdItem), i32, vp, sz, vp]),
        "qlora_last_device_status": (i32, [vp, i32]),
        "nf4_kernel_launch_count": (i64, []),
        "qlora_debug_wait_timeout": (None, [i32]),
        "nf4_timing_enable": (None, [i32]),
        "nf4_timing_read": (i32, [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _status_str(s: int) -> str:
    try:
        return load().nf4_status_str(s).decode()
    except Exception:  # the library itself may be what failed to load
        return "unknown"


def _check(status: int, where: str):
    if status != NF4_OK:
        raise Nf4Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return NF4_F32
    if dt == torch.bfloat16:
        return NF4_BF16
    if dt == torch.float16:
        return NF4_F16
    raise TypeError(f"unsupported dtype {dt}")


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


@dataclass
class Nf4Tensor:
    """A quantized tensor held in device memory (torch buffers) plus its logical shape."""
    shape: tuple
    double_quant: bool
    packed: torch.Tensor
    absmax: torch.Tensor
    nested_absmax: torch.Tensor = None
    offset: torch.Tensor = None

    @property
    def numel(self) -> int:
        n = 1
        for d in self.shape:
            n *= d
        return n

    def c_struct(self) -> _Nf4Tensor:
        return _Nf4Tensor(self.numel, int(self.double_quant), 0, self.packed.data_ptr(),
                          self.absmax.data_ptr(),
                          None if self.nested_absmax is None else self.nested_absmax.data_ptr(),
                          None if self.offset is None else self.offset.data_ptr())

    def nbytes(self) -> int:
        n = self.packed.numel() + self.absmax.numel() * self.absmax.element_size()
        if self.nested_absmax is not None:
            n += 4 * self.nested_absmax.numel()
        return n

    @staticmethod
    def empty(shape, double_quant=True, device="cuda"):
        lib = load()
        n = 1
        for d in shape:
            n *= d
        nb, nnb = lib.nf4_num_blocks(n), lib.nf4_num_nested(n)
        packed = torch.empty((n + 1) // 2, dtype=torch.uint8, device=device)
        if double_quant:
            return Nf4Tensor(tuple(shape), True, packed,
                             torch.empty(nb, dtype=torch.uint8, device=device),
                             torch.empty(nnb, dtype=torch.float32, device=device),
                             torch.zeros(4, dtype=torch.float32, device=device))  # 16-byte slot, [0] used
        return Nf4Tensor(tuple(shape), False, packed, torch.empty(nb, dtype=torch.float32, device=device))


def code_tables():
    """(nf4[16], dyn8[256]) float32 tables exported by the library."""
    lib = load()
    nf4 = (ctypes.c_float * 16)()
    dyn8 = (ctypes.c_float * 256)()
    lib.nf4_code_tables(nf4, dyn8)
    return list(nf4), list(dyn8)


def nf4_quantize(x: torch.Tensor, double_quant: bool = True, out: Nf4Tensor = None,
                 workspace: torch.Tensor = None, stream=None) -> Nf4Tensor:
    lib = load()
    x = x.contiguous()
    if out is None:
        out = Nf4Tensor.empty(tuple(x.shape), double_quant, x.device)
    need = lib.nf4_quantize_workspace_bytes(x.numel(), int(double_quant))
    ws = workspace if workspace is not None else _workspace(need, x.device)
    cs = out.c_struct()
    _check(lib.nf4_quantize(_ptr(x), _dtype_code(x.dtype), x.numel(), ctypes.byref(cs), _ptr(ws),
                            ws.numel(), _stream(stream)), "nf4_quantize")
    return out


def _quant_items(pairs):
    arr = (_QuantItem * len(pairs))()
    keep = []
    for i, (x, q) in enumerate(pairs):
        cs = q.c_struct()
        keep.append(cs)
        arr[i] = _QuantItem(x.data_ptr(), _dtype_code(x.dtype), x.numel(), ctypes.pointer(cs))
    return arr, keep


def nf4_quantize_batch_workspace_bytes(pairs) -> int:
    """Workspace bytes of nf4_quantize_batch for [(x, out), ...]."""
    arr, _keep = _quant_items(pairs)
    return int(load().nf4_quantize_batch_workspace_bytes(len(pairs), arr))


def nf4_quantize_batch(pairs, workspace: torch.Tensor = None, stream=None):
    """Quantize several tensors in one call: ``pairs`` is [(x, out Nf4Tensor), ...] (x contiguous,
    out preallocated); each out gets what nf4_quantize(x, out=out) gives.  Returns the outs."""
    lib = load()
    arr, _keep = _quant_items(pairs)
    need = lib.nf4_quantize_batch_workspace_bytes(len(pairs), arr)
    ws = workspace if workspace is not None else _workspace(need, pairs[0][0].device)
    _check(lib.nf4_quantize_batch(len(pairs), arr, _ptr(ws), ws.numel(), _stream(stream)), "nf4_quantize_batch")
    return [q for _, q in pairs]


def nf4_quantize_noalloc(x: torch.Tensor, out: Nf4Tensor, stream=None) -> Nf4Tensor:
    """nf4_quantize with the library's fixed scratch instead of a workspace.

    For callers that cannot allocate device memory; ``out`` must be allocated by the
    caller.  Calls share one scratch array per device, so they must not overlap on
    the GPU.  numel above NOALLOC_MAX_NUMEL raises Nf4Error(NF4_ERR_TOO_LARGE).
    """
    lib = load()
    x = x.contiguous()
    cs = out.c_struct()
    _check(lib.nf4_quantize_noalloc(_ptr(x), _dtype_code(x.dtype), x.numel(), ctypes.byref(cs),
                                    _stream(stream)), "nf4_quantize_noalloc")
    return out


def nf4_dequantize(q: Nf4Tensor, dtype=torch.float32, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    lib = load()
    y = out if out is not None else torch.empty(q.shape, dtype=dtype, device=q.packed.device)
    cs = q.c_struct()
    _check(lib.nf4_dequantize(ctypes.byref(cs), _ptr(y), _dtype_code(y.dtype), _stream(stream)),
           "nf4_dequantize")
    return y


def nf4_dequantize_batch(pairs, stream=None):
    """Decode several tensors in one call: ``pairs`` is a list of (Nf4Tensor, output tensor),
    all outputs of one dtype; each output gets exactly what ``nf4_dequantize`` writes."""
    lib = load()
    if not pairs:
        return
    dtypes = {y.dtype for _, y in pairs}
    if len(dtypes) != 1:
        raise ValueError("nf4_dequantize_batch: outputs of one dtype")
    structs = [q.c_struct() for q, _ in pairs]
    items = (_DequantItem * len(pairs))()
    for i, ((q, y), cs) in enumerate(zip(pairs, structs)):
        items[i].w = ctypes.pointer(cs)
        items[i].y = _ptr(y)
    _check(lib.nf4_dequantize_batch(len(pairs), items, _dtype_code(pairs[0][1].dtype), _stream(stream)),
           "nf4_dequantize_batch")


def nf4_embedding_rows(E: Nf4Tensor, ids: torch.Tensor, dtype=torch.float32, out: torch.Tensor = None,
                       stream=None) -> torch.Tensor:
    """Rows ``ids`` (device int64) of the NF4 table E [rows, dim], decoded: [len(ids), dim].

    An id outside [0, rows) yields a zero row and sets the device status word
    (read it with ``device_status``).
    """
    lib = load()
    rows, dim = E.shape
    ids = ids.contiguous()
    n = ids.numel()
    y = out if out is not None else torch.empty((n, dim), dtype=dtype, device=E.packed.device)
    cs = E.c_struct()
    _check(lib.nf4_embedding_rows(ctypes.byref(cs), rows, dim, _ptr(ids) if n else None, n, _ptr(y),
                                  _dtype_code(y.dtype), _stream(stream)), "nf4_embedding_rows")
    return y


def nf4_merge_lora(W: Nf4Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float, mode: int = SCALE_LORA,
                   dtype=torch.float32, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Merged weight deq(W) + s B A ([N, K], fp32 or bf16) of an NF4 base W [N, K] and an adapter."""
    lib = load()
    N, K = W.shape
    r = A.shape[0]
    y = out if out is not None else torch.empty((N, K), dtype=dtype, device=W.packed.device)
    cs = W.c_struct()
    _check(lib.nf4_merge_lora(N, K, r, ctypes.c_float(alpha), mode, ctypes.byref(cs), _ptr(A), _ptr(B),
                              _ptr(y), _dtype_code(y.dtype), _stream(stream)), "nf4_merge_lora")
    return y


def qlora_linear_fwd(x: torch.Tensor, W: Nf4Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                     mode: int = SCALE_LORA, y: torch.Tensor = None, T: torch.Tensor = None,
                     workspace: torch.Tensor = None, stream=None):
    """y = x W^T + s (x A^T) B^T; returns (y, T).  x is [M, K] in the compute dtype."""
    lib = load()
    M, K = x.shape
    N = W.shape[0]
    r = A.shape[0]
    cd = _dtype_code(x.dtype)
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if T is None:
        T = torch.empty((M, r), dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else _workspace(
        lib.qlora_fwd_workspace_bytes(M, N, K, r, cd), x.device)
    cs = W.c_struct()
    _check(lib.qlora_linear_fwd(M, N, K, r, ctypes.c_float(alpha), mode, cd, _ptr(x), ctypes.byref(cs),
                                _ptr(A), _ptr(B), _ptr(y), _ptr(T), _ptr(ws), ws.numel(), _stream(stream)),
           "qlora_linear_fwd")
    return y, T


def qlora_linear_fwd_batch(items, workspace: torch.Tensor = None, stream=None):
    """Forward of several projections sharing M: ``items`` is a list of dicts with keys x, A, B,
    alpha, W (an Nf4Tensor) or w16 (the decoded weight), and optionally mode, y, T (as for
    qlora_linear_fwd / qlora_linear_fwd_w16).  Returns [(y, T), ...]; each item equals its
    single call.  Consecutive items that pass the same x tensor share one T pass."""
    lib = load()
    n = len(items)
    M = items[0]["x"].shape[0]
    cd = _dtype_code(items[0]["x"].dtype)
    arr = (_FwdItem * n)()
    keep = []
    outs = []
    for i, it in enumerate(items):
        x, A, B = it["x"], it["A"], it["B"]
        W = it.get("W")
        w16 = it.get("w16")
        N, K = (w16 if w16 is not None else W).shape
        r = A.shape[0]
        y = it.get("y")
        T = it.get("T")
        if y is None:
            y = torch.empty((M, N), dtype=x.dtype, device=x.device)
        if T is None:
            T = torch.empty((M, r), dtype=torch.float32, device=x.device)
        cs = W.c_struct() if W is not None else None
        keep.append(cs)
        arr[i] = _FwdItem(N, K, r, float(it["alpha"]), int(it.get("mode", SCALE_LORA)),
                          ctypes.pointer(cs) if cs is not None else None, A.data_ptr(), B.data_ptr(),
                          x.data_ptr(), y.data_ptr(), T.data_ptr(), w16.data_ptr() if w16 is not None else None)
        outs.append((y, T))
    ws = workspace if workspace is not None else _workspace(
        lib.qlora_fwd_batch_workspace_bytes(M, n, arr, cd), items[0]["x"].device)
    _check(lib.qlora_linear_fwd_batch(M, n, arr, cd, _ptr(ws), ws.numel(), _stream(stream)), "qlora_linear_fwd_batch")
    return outs


def _x_ids(n, xs):
    # stand-in x addresses for workspace queries (never dereferenced): equal ids share an x
    ids = list(range(n)) if xs is None else list(xs)
    first = {}
    return [16 * (1 + first.setdefault(v, len(first))) for v in ids]


def qlora_fwd_batch_workspace_bytes(M: int, shapes, rank: int, dtype=torch.bfloat16, xs=None,
                                    w16: bool = False) -> int:
    """Workspace bytes of qlora_linear_fwd_batch for items of the given (N, K) shapes and rank.
    ``xs``: one hashable per item, equal where items pass the same x (default: all distinct);
    ``w16``: the items give their weights decoded."""
    lib = load()
    arr = (_FwdItem * len(shapes))()
    xid = _x_ids(len(shapes), xs)
    for i, (N, K) in enumerate(shapes):
        arr[i] = _FwdItem(N, K, rank, 1.0, SCALE_LORA, None, None, None, xid[i], None, None, 16 if w16 else None)
    return int(lib.qlora_fwd_batch_workspace_bytes(M, len(shapes), arr, _dtype_code(dtype)))


def qlora_linear_bwd(dy: torch.Tensor, x: torch.Tensor, T: torch.Tensor, W: Nf4Tensor, A: torch.Tensor,
                     B: torch.Tensor, alpha: float, mode: int = SCALE_LORA, dx: torch.Tensor = None,
                     dA: torch.Tensor = None, dB: torch.Tensor = None, workspace: torch.Tensor = None,
                     stream=None):
    """Returns (dX, dA, dB) for the frozen-base QLoRA linear."""
    lib = load()
    M, K = x.shape
    N = W.shape[0]
    r = A.shape[0]
    cd = _dtype_code(x.dtype)
    if dx is None:
        dx = torch.empty((M, K), dtype=x.dtype, device=x.device)
    if dA is None:
        dA = torch.empty((r, K), dtype=torch.float32, device=x.device)
    if dB is None:
        dB = torch.empty((N, r), dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else _workspace(
        lib.qlora_bwd_workspace_bytes(M, N, K, r, cd), x.device)
    cs = W.c_struct()
    _check(lib.qlora_linear_bwd(M, N, K, r, ctypes.c_float(alpha), mode, cd, _ptr(dy), _ptr(x), _ptr(T),
                                ctypes.byref(cs), _ptr(A), _ptr(B), _ptr(dx), _ptr(dA), _ptr(dB),
                                _ptr(ws), ws.numel(), _stream(stream)), "qlora_linear_bwd")
    return dx, dA, dB


def qlora_linear_fwd_w16(x: torch.Tensor, w16: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                         mode: int = SCALE_LORA, y: torch.Tensor = None, T: torch.Tensor = None,
                         workspace: torch.Tensor = None, stream=None):
    """qlora_linear_fwd with the weight given decoded: ``w16`` [N, K] in x's dtype (bf16 or
    half) as nf4_dequantize writes it.  Returns (y, T)."""
    lib = load()
    M, K = x.shape
    N = w16.shape[0]
    r = A.shape[0]
    cd = _dtype_code(x.dtype)
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if T is None:
        T = torch.empty((M, r), dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else _workspace(
        lib.qlora_fwd_w16_workspace_bytes(M, N, K, r, cd), x.device)
    _check(lib.qlora_linear_fwd_w16(M, N, K, r, ctypes.c_float(alpha), mode, cd, _ptr(x), _ptr(w16), _ptr(A),
                                    _ptr(B), _ptr(y), _ptr(T), _ptr(ws), ws.numel(), _stream(stream)),
           "qlora_linear_fwd_w16")
    return y, T


def qlora_linear_bwd_w16(dy: torch.Tensor, x: torch.Tensor, T: torch.Tensor, w16: torch.Tensor, A: torch.Tensor,
                         B: torch.Tensor, alpha: float, mode: int = SCALE_LORA, dx: torch.Tensor = None,
                         dA: torch.Tensor = None, dB: torch.Tensor = None, workspace: torch.Tensor = None,
                         stream=None):
    """qlora_linear_bwd with the weight given decoded (as qlora_linear_fwd_w16).  Returns
    (dX, dA, dB)."""
    lib = load()
    M, K = x.shape
    N = w16.shape[0]
    r = A.shape[0]
    cd = _dtype_code(x.dtype)
    if dx is None:
        dx = torch.empty((M, K), dtype=x.dtype, device=x.device)
    if dA is None:
        dA = torch.empty((r, K), dtype=torch.float32, device=x.device)
    if dB is None:
        dB = torch.empty((N, r), dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else _workspace(
        lib.qlora_bwd_w16_workspace_bytes(M, N, K, r, cd), x.device)
    _check(lib.qlora_linear_bwd_w16(M, N, K, r, ctypes.c_float(alpha), mode, cd, _ptr(dy), _ptr(x), _ptr(T),
                                    _ptr(w16), _ptr(A), _ptr(B), _ptr(dx), _ptr(dA), _ptr(dB), _ptr(ws),
                                    ws.numel(), _stream(stream)), "qlora_linear_bwd_w16")
    return dx, dA, dB


def qlora_linear_bwd_batch(items, workspace: torch.Tensor = None, stream=None):
    """Backward of several projections sharing M: ``items`` is a list of dicts with keys dy, x,
    T, A, B, alpha, W (an Nf4Tensor) or w16 (the decoded weight), and optionally mode, dx, dA,
    dB.  Returns [(dX, dA, dB), ...]; each item equals its single qlora_linear_bwd (or _w16)."""
    lib = load()
    n = len(items)
    M = items[0]["x"].shape[0]
    cd = _dtype_code(items[0]["x"].dtype)
    arr = (_BwdItem * n)()
    keep, outs = [], []
    for i, it in enumerate(items):
        x, A, B = it["x"], it["A"], it["B"]
        K = x.shape[1]
        N = it["dy"].shape[1]
        r = A.shape[0]
        dx = it.get("dx")
        dA = it.get("dA")
        dB = it.get("dB")
        if dx is None:
            dx = torch.empty((M, K), dtype=x.dtype, device=x.device)
        if dA is None:
            dA = torch.empty((r, K), dtype=torch.float32, device=x.device)
        if dB is None:
            dB = torch.empty((N, r), dtype=torch.float32, device=x.device)
        W = it.get("W")
        cs = W.c_struct() if W is not None else None
        keep.append(cs)
        w16 = it.get("w16")
        arr[i] = _BwdItem(N, K, r, float(it["alpha"]), int(it.get("mode", SCALE_LORA)),
                          ctypes.pointer(cs) if cs is not None else None,
                          w16.data_ptr() if w16 is not None else None, A.data_ptr(), B.data_ptr(),
                          it["dy"].data_ptr(), x.data_ptr(), it["T"].data_ptr(), dx.data_ptr(), dA.data_ptr(),
                          dB.data_ptr())
        outs.append((dx, dA, dB))
    ws = workspace if workspace is not None else _workspace(
        lib.qlora_bwd_batch_workspace_bytes(M, n, arr, cd), items[0]["x"].device)
    _check(lib.qlora_linear_bwd_batch(M, n, arr, cd, _ptr(ws), ws.numel(), _stream(stream)), "qlora_linear_bwd_batch")
    return outs


def qlora_bwd_batch_workspace_bytes(M: int, shapes, rank: int, dtype=torch.bfloat16, xs=None,
                                    w16: bool = False) -> int:
    """Workspace bytes of qlora_linear_bwd_batch for items of the given (N, K) shapes and rank
    (``xs`` and ``w16`` as for qlora_fwd_batch_workspace_bytes)."""
    lib = load()
    arr = (_BwdItem * len(shapes))()
    xid = _x_ids(len(shapes), xs)
    for i, (N, K) in enumerate(shapes):
        arr[i] = _BwdItem(N, K, rank, 1.0, SCALE_LORA, None, 16 if w16 else None, None, None, None, xid[i], None,
                          None, None, None)
    return int(lib.qlora_bwd_batch_workspace_bytes(M, len(shapes), arr, _dtype_code(dtype)))


def debug_wait_timeout(on: bool = True):
    """Arm (or disarm) the library's test of its timeout path: the next tensor-core contraction
    runs with a 20 ms wait limit and its first CTA leaves its first stage unissued, so that
    launch ends with NF4_ERR_TIMEOUT in the device status word (its outputs unspecified)."""
    load().qlora_debug_wait_timeout(int(on))


def device_status(clear: bool = True, stream=None) -> int:
    return int(load().qlora_last_device_status(_stream(stream), int(clear)))


def launch_count() -> int:
    return int(load().nf4_kernel_launch_count())


def timing_enable(on: bool = True):
    """Turn the library's per-kernel event timing on or off."""
    load().nf4_timing_enable(int(on))


def timing_read(kind: int, reset: bool = True):
    """(total milliseconds, launches) of one timed kernel kind since the last reset."""
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    _check(load().nf4_timing_read(kind, ctypes.byref(ms), ctypes.byref(n), int(reset)), "nf4_timing_read")
    return ms.value, n.value
