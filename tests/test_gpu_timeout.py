"""The timeout path of the bounded device waits, exercised without faulting the GPU.

qlora_debug_wait_timeout arms one launch: its first CTA leaves its first pipeline stage
unissued and the launch runs with a 20 ms wait limit, so the waits for that stage run out.
The launch must return, report NF4_ERR_TIMEOUT through the device status word, free what it
holds (TMEM, copies in flight), and leave the context usable: the next call of the same
entry point matches the oracle element by element.
"""

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


def _case(M, N, K, r, seed):
    ref = onf4.quantize(wl.normal((N, K), 0.02, 8, seed), double_quant=True)
    q = binding.Nf4Tensor.empty((N, K), True, DEV)
    q.packed.copy_(torch.from_numpy(ref["packed"]))
    q.absmax.copy_(torch.from_numpy(ref["absmax"]))
    q.nested_absmax.copy_(torch.from_numpy(ref["nested"]))
    q.offset[0] = float(ref["offset"])
    x = onf4.round_bf16(wl.normal((M, K), 1.0, 8, seed + 1))
    A, B = wl.adapters(N, K, r, 8, seed + 2)
    w64 = onf4.round_bf16(onf4.dequantize(ref, "f32")).reshape(N, K).astype(np.float64)
    return q, x, A, B, w64


def _forward_matches_oracle(q, x, A, B, w64, alpha, r):
    xd = torch.from_numpy(x).to(DEV).bfloat16()
    y, T = binding.qlora_linear_fwd(xd, q, torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV), alpha)
    torch.cuda.synchronize()
    s = qlora.lora_scale(alpha, r)
    y_ref, T_ref = qlora.forward(x, w64, A, B, s, "bf16")
    b = parity.forward_bounds(x, w64, A, B, s, "bf16", y_ref, T_ref)
    parity.check(dict(y=y.float().cpu().numpy(), T=T.cpu().numpy()), dict(y=y_ref, T=T_ref), b, "bf16")


@pytest.mark.parametrize("M", [4, 300], ids=["small-M weight pass", "tiled GEMM"])
def test_wait_runs_out_then_the_next_call_is_clean(lib, M):
    N, K, r, alpha = 520, 1024, 8, 16.0
    q, x, A, B, w64 = _case(M, N, K, r, 40 + M)
    assert binding.device_status(clear=True) == binding.NF4_OK
    binding.debug_wait_timeout(True)
    xd = torch.from_numpy(x).to(DEV).bfloat16()
    binding.qlora_linear_fwd(xd, q, torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV), alpha)
    torch.cuda.synchronize()
    assert binding.device_status(clear=True) == binding.NF4_ERR_TIMEOUT
    # the switch is one-shot: the next launch runs with the normal limit and every stage
    _forward_matches_oracle(q, x, A, B, w64, alpha, r)
    assert binding.device_status(clear=True) == binding.NF4_OK


def test_disarming_the_switch(lib):
    q, x, A, B, w64 = _case(4, 264, 512, 4, 77)
    binding.debug_wait_timeout(True)
    binding.debug_wait_timeout(False)
    _forward_matches_oracle(q, x, A, B, w64, 8.0, 4)
    assert binding.device_status(clear=True) == binding.NF4_OK
