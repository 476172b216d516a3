"""GPU parity of nf4_quantize / nf4_dequantize against the oracle (bit-exact).

Inputs come from the seeded generators in bit_nf4_quantized_gb300.workloads; the
same bytes go to the CUDA path (through the C ABI) and to the oracle.
"""

import numpy as np
import pytest
import torch

from bit_nf4_quantized_gb300 import binding
from bit_nf4_quantized_gb300 import workloads as wl
from oracle import codebooks as cb
from oracle import nf4 as onf4

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _to_device(x32: np.ndarray, dtype):
    t = torch.from_numpy(x32).to(DEV)
    return t.to(dtype)


def _host_values(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def _assert_same_quant(q_gpu, q_ref):
    assert np.array_equal(q_gpu.packed.cpu().numpy(), q_ref["packed"])
    if q_ref["double_quant"]:
        assert np.array_equal(q_gpu.absmax.cpu().numpy(), q_ref["absmax"])
        assert np.array_equal(q_gpu.nested_absmax.cpu().numpy().view(np.uint32),
                              q_ref["nested"].view(np.uint32))
        assert q_gpu.offset[0].cpu().numpy().view(np.uint32) == np.float32(q_ref["offset"]).view(np.uint32)
    else:
        assert np.array_equal(q_gpu.absmax.cpu().numpy().view(np.uint32), q_ref["absmax"].view(np.uint32))


SIZES = [1, 2, 3, 63, 64, 65, 127, 129, 1000, 16383, 16384, 16385, 64 * 256 * 3 + 17, 2 ** 20 + 7 * 16384]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dq", [True, False])
def test_quantize_bit_exact(lib, n, dtype, dq):
    x = wl.normal(n, 0.02, 5, n % 1000)
    if n > 200:
        x = wl.with_outliers(x, 0.001, 50.0, 5, 500)
    xd = _to_device(x, dtype)
    q = binding.nf4_quantize(xd, double_quant=dq)
    ref = onf4.quantize(_host_values(xd), double_quant=dq)
    _assert_same_quant(q, ref)
    assert binding.device_status() == binding.NF4_OK


def test_quantize_near_every_threshold(lib):
    """Values whose quotient x/a lands within a few ulps of each midpoint between
    neighbouring NF4 values, under block maxima that are not powers of two (so that
    x * RN(1/a) and RN(x/a) can round differently): codes must be those of the IEEE
    quotient, as the oracle's exact nearest-value search takes them."""
    nf4 = cb.nf4_codebook().astype(np.float64)
    mids = (nf4[:-1] + nf4[1:]) / 2
    rng = np.random.default_rng(11)
    blocks = []
    for _ in range(256):
        a = np.float32(rng.uniform(0.5, 2.0) * 2.0 ** int(rng.integers(-20, 20)))
        probes = []
        for m in mids:
            v0 = np.float32(m * np.float64(a))
            for k in range(-3, 4):
                v = v0
                for _ in range(abs(k)):
                    v = np.nextafter(v, np.float32(np.inf if k > 0 else -np.inf))
                probes.append(min(max(v, -a), a))
        probes = rng.permutation(np.array(probes, np.float32))
        for c0 in range(0, len(probes), 63):   # every block: its maximum a, then 63 probes
            chunk = probes[c0:c0 + 63]
            blocks.append(np.concatenate([[a], chunk, np.zeros(63 - len(chunk), np.float32)]))
    x = np.concatenate(blocks).astype(np.float32)
    xd = _to_device(x, torch.float32)
    q = binding.nf4_quantize(xd, double_quant=False)
    ref = onf4.quantize(_host_values(xd), double_quant=False)
    _assert_same_quant(q, ref)
    assert binding.device_status() == binding.NF4_OK


def test_quantize_bf16_every_ratio(lib):
    """bf16 input: every quotient of two bf16 values that the encoder's bf16 path decides
    from one fused multiply-add.  Each block holds its maximum a and 63 values x; a runs
    over all 128 bf16 significands at binary exponents inside the range where 1/a is normal
    (-126 .. 125) and outside it (126, 127, and subnormal a); x runs over all significands
    at a*2^-d, d = 0..17, both signs.  The codes must be the oracle's, which divides."""
    sig = 1.0 + np.arange(128) / 128.0
    rng = np.random.default_rng(5)
    blocks = []
    for ea in (-126, -70, -3, 0, 7, 88, 125, 126, 127, -127, -131):
        for ma in sig:
            a = np.float32(ma * 2.0 ** ea)
            xs = np.concatenate([sgn * sig * 2.0 ** (ea - d) for d in range(18) for sgn in (1.0, -1.0)])
            xs = xs[np.abs(xs) <= np.float64(a)].astype(np.float32)
            xs = rng.permutation(xs)
            for c0 in range(0, xs.size, 63):
                chunk = xs[c0:c0 + 63]
                blocks.append(np.concatenate([[a], chunk, np.zeros(63 - chunk.size, np.float32)]))
    x = np.concatenate(blocks).astype(np.float32)
    xd = _to_device(x, torch.bfloat16)
    xh = _host_values(xd)
    # the block maxima survive the rounding to bf16 as maxima
    assert np.array_equal(onf4.block_absmax(xh), np.abs(xh[0::64]))
    for dq in (False, True):
        q = binding.nf4_quantize(xd, double_quant=dq)
        _assert_same_quant(q, onf4.quantize(xh, double_quant=dq))
    assert binding.device_status() == binding.NF4_OK


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_16_byte_aligned_view(lib, dtype):
    """An input 16 but not 32 bytes aligned takes the 16-byte loads; same bytes as the oracle."""
    n = 3 * 16384 + 1000
    per16 = 16 // torch.tensor([], dtype=dtype).element_size()
    big = wl.device_normal((n + per16,), 0.02, wl.seed_for(5, 77), DEV, dtype)
    x = big[per16:]
    assert x.data_ptr() % 32 == 16
    for dq in (True, False):
        q = binding.nf4_quantize(x, double_quant=dq)
        _assert_same_quant(q, onf4.quantize(_host_values(x), double_quant=dq))
    assert binding.device_status() == binding.NF4_OK


@pytest.mark.parametrize("n", [2 ** 26, 2 ** 26 + 16384])
def test_quantize_offset_at_a_power_of_two_group_count(lib, n):
    """4096 groups of 256 blocks (the offset tree is exactly the 4096 group sums) and one
    group more (the tree pads to 8192 with zeros): the offset, which the block pass's last
    CTA computes, and the nested maxima and codes (sampled groups) are the oracle's; bf16
    input."""
    x = wl.device_normal((n,), 0.02, wl.seed_for(5, n % 1000), DEV, torch.bfloat16)
    q = binding.nf4_quantize(x)
    x_host = _host_values(x)
    ng = -(-n // 16384)
    _sampled_groups_check(x_host, q, [0, 1, ng // 2, ng - 2, ng - 1])
    assert binding.device_status() == binding.NF4_OK


def test_quantize_batch_equals_single_calls(lib):
    """nf4_quantize_batch over 11 tensors (bf16 and fp32, with and without double quantization,
    ragged sizes; more than 8, so the items run in several launches) gives every tensor the
    bytes a single nf4_quantize call gives, and those are the oracle's."""
    specs = [(torch.bfloat16, True, 16384 * 5 + 3), (torch.bfloat16, False, 1000), (torch.bfloat16, True, 64),
             (torch.float32, True, 16384 * 3), (torch.float32, False, 77777), (torch.float32, True, 1),
             (torch.bfloat16, True, 4096 * 1024), (torch.bfloat16, True, 129), (torch.bfloat16, False, 65),
             (torch.bfloat16, True, 300000), (torch.bfloat16, True, 16385)]
    pairs, singles = [], []
    for i, (dt, dq, n) in enumerate(specs):
        x = wl.device_normal((n,), 0.02, wl.seed_for(5, 500 + i), DEV, dt)
        pairs.append((x, binding.Nf4Tensor.empty((n,), dq, DEV)))
        singles.append(binding.nf4_quantize(x, dq))
    binding.nf4_quantize_batch(pairs)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    for (x, q), one, (dt, dq, n) in zip(pairs, singles, specs):
        assert torch.equal(q.packed, one.packed)
        assert torch.equal(q.absmax.view(torch.uint8), one.absmax.view(torch.uint8))
        if dq:
            assert torch.equal(q.nested_absmax.view(torch.int32), one.nested_absmax.view(torch.int32))
            assert torch.equal(q.offset.view(torch.int32), one.offset.view(torch.int32))
        if n <= 100000:
            _assert_same_quant(q, onf4.quantize(_host_values(x), double_quant=dq))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
def test_dequantize_batch_equals_single_calls(lib, dtype):
    """nf4_dequantize_batch over 10 tensors (with and without double quantization, ragged
    sizes; more than 8, so two runs of launches) writes every output exactly as a single
    nf4_dequantize call does, and those are the oracle's values."""
    odt = {torch.bfloat16: "bf16", torch.float32: "f32", torch.float16: "f16"}[dtype]
    sizes = [(16384 * 5 + 3, True), (1000, False), (64, True), (16384 * 3, True), (77777, False),
             (1, True), (4096 * 1024, True), (129, True), (65, False), (300000, True)]
    xs, pairs, singles = [], [], []
    for i, (n, dq) in enumerate(sizes):
        x = wl.device_normal((n,), 0.02, wl.seed_for(5, 700 + i), DEV, torch.bfloat16)
        q = binding.nf4_quantize(x, dq)
        xs.append(x)
        pairs.append((q, torch.full((n,), float("nan"), dtype=dtype, device=DEV)))
        singles.append(binding.nf4_dequantize(q, dtype))
    binding.nf4_dequantize_batch(pairs)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    for (q, y), one, x, (n, dq) in zip(pairs, singles, xs, sizes):
        assert torch.equal(y.view(torch.int16 if dtype != torch.float32 else torch.int32),
                           one.view(torch.int16 if dtype != torch.float32 else torch.int32))
        if n <= 100000:
            want = onf4.dequantize(onf4.quantize(_host_values(x), double_quant=dq), odt)
            assert np.array_equal(y.float().cpu().numpy().view(np.uint32), want.astype(np.float32).view(np.uint32))


def test_quantize_ticket_counters_wrap(lib):
    """The block pass's ticket counters come from the library's pool of 16384 that every call
    puts back to zero: 16500 double-quant calls in a row (every counter used again) all give the
    oracle's offset."""
    x = wl.device_normal((16384 * 2 + 5,), 0.02, wl.seed_for(5, 600), DEV, torch.bfloat16)
    ref = onf4.quantize(_host_values(x), double_quant=True)
    q = binding.Nf4Tensor.empty(tuple(x.shape), True, DEV)
    ws = torch.empty(binding.load().nf4_quantize_workspace_bytes(x.numel(), 1), dtype=torch.uint8, device=DEV)
    offsets = torch.empty(16500, dtype=torch.float32, device=DEV)
    for i in range(16500):
        binding.nf4_quantize(x, True, out=q, workspace=ws)
        offsets[i:i + 1].copy_(q.offset[:1])
    torch.cuda.synchronize()
    assert binding.device_status() == binding.NF4_OK
    want = np.float32(ref["offset"]).view(np.uint32)
    assert np.all(offsets.cpu().numpy().view(np.uint32) == want)
    _assert_same_quant(q, ref)


def test_quantize_special_blocks(lib):
    nf4 = cb.nf4_codebook()
    x = np.zeros(64 * 300 + 5, np.float32)
    # block 0: exact code multiples and exact ties at absmax 1
    x[0] = 1.0
    x[1:17] = nf4
    mids = [(nf4[j] + nf4[j + 1]) / np.float32(2) for j in range(15)]
    x[17:32] = np.array(mids, np.float32)
    # block 1 stays all zero; block 2 has -0.0 and one tiny subnormal
    x[128:192] = -0.0
    x[150] = 1e-44
    # block 3: the maximum is negative
    x[192:256] = np.linspace(-3, 1, 64, dtype=np.float32)
    for dq in (True, False):
        xd = torch.from_numpy(x).to(DEV)
        q = binding.nf4_quantize(xd, double_quant=dq)
        _assert_same_quant(q, onf4.quantize(x, double_quant=dq))


def _group_of_maxima(maxima: np.ndarray, seed: int) -> np.ndarray:
    """One nested group (256 blocks of 64) whose block b has the largest magnitude maxima[b]:
    that value at a seeded position of the block, with a seeded sign, the other entries of
    the block smaller in magnitude."""
    rng = np.random.default_rng(seed)
    x = (rng.uniform(-1.0, 1.0, (256, 64)) * maxima[:, None].astype(np.float64) * 0.999).astype(np.float32)
    pos = rng.integers(0, 64, 256)
    sign = np.where(rng.integers(0, 2, 256) == 1, np.float32(-1.0), np.float32(1.0))
    x[np.arange(256), pos] = maxima * sign
    return x.reshape(-1)


def _maxima_with_exponents(lo: int, hi: int, seed: int) -> np.ndarray:
    """256 fp32 values with biased exponents spread over [lo, hi] (both ends present) and
    seeded 23-bit fractions."""
    rng = np.random.default_rng(seed)
    e = rng.integers(lo, hi + 1, 256).astype(np.uint32)
    e[0], e[1] = lo, hi
    frac = rng.integers(0, 1 << 23, 256).astype(np.uint32)
    return ((e << 23) | frac).view(np.float32)


def test_quantize_group_sum_regimes(lib):
    """The block pass forms a group's sum of maxima exactly in integers when the maxima's
    exponents span at most 21 binades, else by the float64 tree; both must give the oracle's
    float64 tree result.  One-group tensors (offset = that sum / 256, rounded to fp32) and a
    tensor of all of them: exponent spans 0, 21 (the last exact case) and 22, 30 (tree), all
    subnormal maxima, subnormal next to the smallest normals, zero and non-zero blocks mixed,
    and the near-equal maxima of real weights."""
    groups = {
        "span0": _maxima_with_exponents(120, 120, 1),
        "span21": _maxima_with_exponents(100, 121, 2),
        "span22": _maxima_with_exponents(100, 122, 3),
        "span30": _maxima_with_exponents(97, 127, 4),
        "subnormal": (np.random.default_rng(5).integers(1, 1 << 23, 256).astype(np.uint32)).view(np.float32),
        "subnormal_and_min_normal": _maxima_with_exponents(0, 1, 6),
        "zeros_mixed": np.where(np.arange(256) % 3 == 0, np.float32(0.0), _maxima_with_exponents(110, 125, 7)),
        "weights": np.abs(wl.normal(256, 0.05, 5, 77)) + np.float32(0.05),
    }
    parts = []
    for i, (name, m) in enumerate(groups.items()):
        x = _group_of_maxima(m.astype(np.float32), 100 + i)
        parts.append(x)
        for dtype in (torch.float32,):
            xd = _to_device(x, dtype)
            q = binding.nf4_quantize(xd, double_quant=True)
            _assert_same_quant(q, onf4.quantize(_host_values(xd), double_quant=True))
    x = np.concatenate(parts)
    xd = _to_device(x, torch.float32)
    q = binding.nf4_quantize(xd, double_quant=True)
    _assert_same_quant(q, onf4.quantize(x, double_quant=True))
    assert binding.device_status() == binding.NF4_OK


def test_quantize_is_deterministic(lib):
    x = _to_device(wl.normal(64 * 256 * 40 + 3, 0.02, 5, 900), torch.float32)
    a = binding.nf4_quantize(x)
    b = binding.nf4_quantize(x)
    for f in ("packed", "absmax", "nested_absmax"):
        assert torch.equal(getattr(a, f), getattr(b, f))
    assert torch.equal(a.offset[:1], b.offset[:1])


def test_nonfinite_sets_device_status(lib):
    binding.device_status(clear=True)
    for bad in (float("nan"), float("inf")):
        x = torch.zeros(5000, device=DEV)
        x[1234] = bad
        binding.nf4_quantize(x)
        assert binding.device_status(clear=True) == binding.NF4_ERR_NONFINITE
    binding.nf4_quantize(torch.ones(5000, device=DEV))
    assert binding.device_status(clear=True) == binding.NF4_OK


def _upload(ref, shape):
    """The oracle's quantized tensor copied to the device (so dequant is tested on its own)."""
    q = binding.Nf4Tensor.empty(shape, ref["double_quant"], DEV)
    q.packed.copy_(torch.from_numpy(ref["packed"]))
    q.absmax.copy_(torch.from_numpy(ref["absmax"]))
    if ref["double_quant"]:
        q.nested_absmax.copy_(torch.from_numpy(ref["nested"]))
        q.offset[0] = float(ref["offset"])
    return q


@pytest.mark.parametrize("n", [1, 5, 64, 65, 1000, 16385, 64 * 256 * 5 + 33, 2 ** 20 + 7 * 16384])
@pytest.mark.parametrize("dq", [True, False])
def test_dequantize_bit_exact(lib, n, dq):
    x = wl.student_t(n, 5, 0.02, 5, 7)
    ref = onf4.quantize(x, double_quant=dq)
    q = _upload(ref, (n,))
    for dtype, odt in ((torch.float32, "f32"), (torch.bfloat16, "bf16"), (torch.float16, "f16")):
        y = binding.nf4_dequantize(q, dtype)
        want = onf4.dequantize(ref, odt)
        got = y.float().cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def _sampled_groups_check(x_host: np.ndarray, q, groups):
    """Check selected 16384-element groups of a large quantization against the oracle's steps."""
    a = onf4.block_absmax(x_host)
    offset = onf4.absmax_offset(a)
    assert q.offset[0].cpu().numpy().view(np.uint32) == np.float32(offset).view(np.uint32)
    packed = q.packed.cpu().numpy()
    codes = q.absmax.cpu().numpy()
    nested = q.nested_absmax.cpu().numpy()
    dyn8 = cb.dynamic8_codebook()
    nb = a.size
    for g in groups:
        e0, e1 = g * 16384, min((g + 1) * 16384, x_host.size)
        part = onf4.quantize(x_host[e0:e1], double_quant=False)
        assert np.array_equal(packed[e0 // 2:(e1 + 1) // 2], part["packed"])
        b0, b1 = g * 256, min((g + 1) * 256, nb)
        c = (a[b0:b1] - offset).astype(np.float32)
        na = np.float32(np.max(np.abs(c)))
        assert nested[g] == na
        want = onf4.nearest_code(c / na, dyn8) if na > 0 else np.full(c.size, 127, np.uint8)
        assert np.array_equal(codes[b0:b1], want)


@pytest.mark.parametrize("log2n", [24, 28])
def test_quantize_large_sampled(lib, log2n):
    n = 2 ** log2n
    x = wl.device_normal((n,), 0.02, wl.seed_for(5, log2n), DEV, torch.float32)
    q = binding.nf4_quantize(x)
    x_host = x.cpu().numpy()
    ng = n // 16384
    groups = sorted(set([0, 1, ng // 2, ng - 1] + list(np.random.default_rng(log2n).integers(0, ng, 6))))
    _sampled_groups_check(x_host, q, groups)
    # dequantized values of the sampled groups, bf16 output
    y = binding.nf4_dequantize(q, torch.bfloat16)
    ys = y.float().cpu().numpy()
    ref_full = dict(numel=n, double_quant=True, packed=q.packed.cpu().numpy(), absmax=q.absmax.cpu().numpy(),
                    nested=q.nested_absmax.cpu().numpy(), offset=q.offset[0].cpu().numpy())
    for g in groups[:4]:
        sub = dict(ref_full)
        e0, e1 = g * 16384, (g + 1) * 16384
        sub.update(numel=e1 - e0, packed=ref_full["packed"][e0 // 2:e1 // 2],
                   absmax=ref_full["absmax"][g * 256:(g + 1) * 256], nested=ref_full["nested"][g:g + 1])
        want = onf4.dequantize(sub, "bf16")
        assert np.array_equal(ys[e0:e1].view(np.uint32), want.view(np.uint32))
