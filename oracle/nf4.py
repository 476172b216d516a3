"""NF4 blockwise quantization with nested (double) quantization: plain CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What it computes, step by step, in the order of [ADAPT] section "Packed NF4 and the
portable QLoRA profile" (with the block sizes of [QUAL-2] key ``nf4``):

1. The flattened tensor is cut into 64-element blocks (the last may be short;
   elements past ``numel`` take no part).  a_b = max |x_i| over the block.
2. v_i = x_i / a_b, one IEEE float32 division (round to nearest even).  The 4-bit
   code is the index of the NF4 value nearest to v_i; an exact tie goes to the
   lower index.  A block with a_b = 0 gets the code of 0.0 for every element.
3. Two codes per byte: element 2i in the high nibble, 2i+1 in the low nibble; a
   trailing odd element leaves the low nibble 0.
4. Double quantization ("centered by their global FP32 mean and quantized with the
   signed dynamic8 codebook in 256 element blocks"):
   offset = mean of all a_b, summed in float64 by a fixed pairwise tree (within
   each 256-group: s[i] += s[i + h] for h = 128, 64, ..., 1, missing entries 0;
   then the same tree over the group sums padded with zeros to a power of two)
   and rounded once to float32 after dividing by the block count.
   c_b = a_b - offset (float32); per 256-group na = max |c_b|; the 8-bit code is
   the dynamic8 value nearest to c_b / na (float32 division; ties to the lower
   index; na = 0 gives the code of 0.0).
5. Dequantization ([ADAPT] "Fused GPU NF4 decodes inside the matrix kernel"; the
   separately rounded decode of [QUAL] ``jit.kernel_identity``):
   a'_b = (dyn8[code_b] * na) + offset as two float32 operations, no fused
   multiply-add; without double quantization a'_b = a_b.  w_i = nf4[q_i] * a'_b
   (one float32 multiply); a bfloat16 output is that value rounded to nearest even.

Storage sizes ([GATE] "P3 is solved": N/2 + N/64 + N/4096 + 4 bytes; [QUAL]
``component_benchmarks.packed_gpu_bytes``): ceil(N/2) packed bytes, ceil(N/64)
absmax codes, 4 * ceil(ceil(N/64)/256) nested bytes, plus a 4-byte offset that the
device copy passes separately.

Readings of points the pages leave open (nibble order, tie rule, fp64 tree for the
mean, no-FMA decode) are listed with the rest of the design notes; the pins for
each step are in tests/test_oracle_nf4.py.
"""

import numpy as np

from .codebooks import dynamic8_codebook, nf4_codebook

BLOCK = 64
NESTED_BLOCK = 256
NF4_ZERO_INDEX = 7


def num_blocks(numel: int) -> int:
    return -(-numel // BLOCK)


def num_nested(numel: int) -> int:
    return -(-num_blocks(numel) // NESTED_BLOCK)


def packed_bytes(numel: int, double_quant: bool = True, with_offset: bool = False) -> int:
    """Bytes of one quantized matrix: packed codes + absmax + nested absmax (+ offset)."""
    nb = num_blocks(numel)
    if not double_quant:
        return -(-numel // 2) + 4 * nb
    return -(-numel // 2) + nb + 4 * num_nested(numel) + (4 if with_offset else 0)


def nearest_code(v: np.ndarray, table: np.ndarray, chunk: int = 1 << 16) -> np.ndarray:
    """Index of the table value nearest to each v (exact float64 distances; ties -> lower index)."""
    v64 = np.asarray(v, dtype=np.float64).ravel()
    t64 = table.astype(np.float64)
    out = np.empty(v64.shape, dtype=np.uint8)
    for s in range(0, v64.size, chunk):
        d = np.abs(v64[s:s + chunk, None] - t64[None, :])
        out[s:s + chunk] = np.argmin(d, axis=1)   # first minimum = lower index on a tie
    return out.reshape(np.shape(v))


def block_absmax(x32: np.ndarray) -> np.ndarray:
    n = x32.size
    nb = num_blocks(n)
    padded = np.zeros(nb * BLOCK, dtype=np.float32)   # zeros never raise a max of |x|
    padded[:n] = np.abs(x32)
    return padded.reshape(nb, BLOCK).max(axis=1)


def _pairwise_tree_sum(vals64: np.ndarray) -> np.float64:
    """s[i] += s[i + h] for h = n/2, ..., 1 over a power-of-two length (zero padded)."""
    n = 1
    while n < vals64.size:
        n *= 2
    s = np.zeros(n, dtype=np.float64)
    s[:vals64.size] = vals64
    while n > 1:
        n //= 2
        s = s[:n] + s[n:2 * n]
    return s[0]


def group_sums(absmax: np.ndarray) -> np.ndarray:
    """Float64 pairwise-tree sum of each 256-group of block absmax values."""
    nb = absmax.size
    ng = -(-nb // NESTED_BLOCK)
    out = np.empty(ng, dtype=np.float64)
    a64 = absmax.astype(np.float64)
    for g in range(ng):
        chunk = np.zeros(NESTED_BLOCK, dtype=np.float64)
        part = a64[g * NESTED_BLOCK:(g + 1) * NESTED_BLOCK]
        chunk[:part.size] = part
        out[g] = _pairwise_tree_sum(chunk)
    return out


def absmax_offset(absmax: np.ndarray) -> np.float32:
    """Global float32 mean of the block absmax values (fixed float64 tree, one final rounding)."""
    total = _pairwise_tree_sum(group_sums(absmax))
    return np.float32(total / np.float64(absmax.size))


def quantize(x, double_quant: bool = True) -> dict:
    """Quantize a float tensor (float32, or bfloat16 values held in float32) to NF4.

    Returns dict(numel, double_quant, packed uint8[ceil(n/2)], absmax (uint8[nb]
    codes with double quantization, else float32[nb]), nested float32[nnb] or None,
    offset float32 or None).  Raises ValueError on empty or non-finite input.
    """
    x32 = np.ascontiguousarray(x, dtype=np.float32).ravel()
    n = x32.size
    if n == 0:
        raise ValueError("empty tensor")
    if not np.all(np.isfinite(x32)):
        raise ValueError("non-finite input")
    nf4 = nf4_codebook()
    nb = num_blocks(n)
    a = block_absmax(x32)                                   # step 1
    a_per_elem = np.repeat(a, BLOCK)[:n]
    q = np.full(n, NF4_ZERO_INDEX, dtype=np.uint8)
    live = a_per_elem > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        v = x32 / a_per_elem                                # step 2: float32 division
    q[live] = nearest_code(v[live], nf4)
    codes = np.zeros(2 * (-(-n // 2)), dtype=np.uint8)      # step 3
    codes[:n] = q
    packed = ((codes[0::2] << 4) | codes[1::2]).astype(np.uint8)
    out = dict(numel=n, double_quant=bool(double_quant), packed=packed,
               absmax=a.astype(np.float32), nested=None, offset=None)
    if not double_quant:
        return out
    dyn8 = dynamic8_codebook()                              # step 4
    offset = absmax_offset(a)
    c = (a - offset).astype(np.float32)
    ng = num_nested(n)
    cpad = np.zeros(ng * NESTED_BLOCK, dtype=np.float32)
    cpad[:nb] = np.abs(c)
    na = cpad.reshape(ng, NESTED_BLOCK).max(axis=1).astype(np.float32)
    na_per_block = np.repeat(na, NESTED_BLOCK)[:nb]
    zero_code = int(np.flatnonzero(dyn8 == 0)[0])
    acode = np.full(nb, zero_code, dtype=np.uint8)
    live = na_per_block > 0
    acode[live] = nearest_code(c[live] / na_per_block[live], dyn8)
    out.update(absmax=acode, nested=na, offset=np.float32(offset))
    return out


def unpack_codes(packed: np.ndarray, numel: int) -> np.ndarray:
    hi = packed >> 4
    lo = packed & 0x0F
    return np.stack([hi, lo], axis=1).ravel()[:numel].astype(np.uint8)


def block_scales(qt: dict) -> np.ndarray:
    """a'_b for every block: dyn8[code] * na + offset (two float32 roundings) or the fp32 absmax."""
    if not qt["double_quant"]:
        return np.asarray(qt["absmax"], dtype=np.float32)
    dyn8 = dynamic8_codebook()
    nb = qt["absmax"].size
    na = np.repeat(qt["nested"].astype(np.float32), NESTED_BLOCK)[:nb]
    prod = (dyn8[qt["absmax"]] * na).astype(np.float32)
    return (prod + np.float32(qt["offset"])).astype(np.float32)


def dequantize(qt: dict, out_dtype: str = "f32") -> np.ndarray:
    """Decode to float32 values; ``out_dtype='bf16'`` or ``'f16'`` returns them rounded once to
    bfloat16 or IEEE half (as float32 values)."""
    n = qt["numel"]
    nf4 = nf4_codebook()
    q = unpack_codes(qt["packed"], n)
    scale = np.repeat(block_scales(qt), BLOCK)[:n]
    w = (nf4[q] * scale).astype(np.float32)
    if out_dtype == "bf16":
        return round_bf16(w)
    if out_dtype == "f16":
        return round_f16(w)
    return w


def round_bf16(x) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returned as float32 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    bias = ((u >> 16) & 1) + 0x7FFF
    r = ((u + bias) & 0xFFFF0000).astype(np.uint32)
    out = r.view(np.float32).copy()
    out[nan] = np.nan
    return out.reshape(np.shape(x))


def round_f16(x) -> np.ndarray:
    """Round float32 values to IEEE binary16 (nearest, ties to even, gradual underflow, overflow to
    infinity; numpy's float32 -> float16 conversion); returned as float32 values."""
    with np.errstate(over="ignore"):   # overflow to infinity is the IEEE result
        return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of bfloat16 values that are held exactly in float32."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
