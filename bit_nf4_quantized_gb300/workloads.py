"""Seeded synthetic inputs and the workload shapes; no NF4 or LoRA arithmetic here.

This module is the only code that both the CUDA-side tests/bench and the oracle's
callers use: it draws random numbers and names shapes, nothing else.

Seeds: numpy PCG64 with seed 71 + 1000 * workload + tensor id (71 is the adapter
seed of "Native model adaptation and NF4", section "Adapter API").  Large tensors
for timing only are drawn on the device with a seeded torch generator.

Distributions: N(0, s) means standard deviation s.  Student-t(5) is drawn from its
definition, z0 / sqrt((z1^2 + ... + z5^2) / 5).
"""

import numpy as np

BASE_SEED = 71

# Workload 1: one 576 x 576 matrix, fp32 profile.
W1 = dict(name="576x576 fp32 QLoRA fwd+bwd, M=512, r=16, alpha=32", N=576, K=576, M=512, r=16,
          alpha=32.0, w_std=0.02, compute="f32")

# Workload 2: SmolLM2-135M-shaped stack (hidden 576, intermediate 1536, 30 layers).
SMOLLM2_LAYER = [("q_proj", 576, 576), ("k_proj", 192, 576), ("v_proj", 192, 576),
                 ("o_proj", 576, 576), ("gate_proj", 1536, 576), ("up_proj", 1536, 576),
                 ("down_proj", 576, 1536)]
W2 = dict(name="SmolLM2-135M-shaped 30-layer stack, QLoRA q,v, M=512, r=16, alpha=32, bf16",
          layers=30, shapes=SMOLLM2_LAYER, targets=("q_proj", "v_proj"), M=512, r=16, alpha=32.0,
          w_std=0.02, compute="bf16")

# Workload 3: one Llama-3-8B-shaped layer (hidden 4096, intermediate 14336).
LLAMA8B_LAYER = [("q_proj", 4096, 4096), ("k_proj", 1024, 4096), ("v_proj", 1024, 4096),
                 ("o_proj", 4096, 4096), ("gate_proj", 14336, 4096), ("up_proj", 14336, 4096),
                 ("down_proj", 4096, 14336)]
# The activation each projection of a transformer layer reads: q, k and v read the attention
# block's normalised input, gate and up the MLP block's, o the attention output, down the MLP's
# gated activation.  Projections that read the same activation get one shared x.
LAYER_INPUTS = {"q_proj": "attn_in", "k_proj": "attn_in", "v_proj": "attn_in", "o_proj": "attn_out",
                "gate_proj": "mlp_in", "up_proj": "mlp_in", "down_proj": "mlp_act"}
W3 = dict(name="Llama-3-8B-shaped layer, 7 QLoRA targets, M=4096 (2x2048), r=16, alpha=16, bf16",
          shapes=LLAMA8B_LAYER, M=4096, r=16, alpha=16.0, w_scale=0.02, t_df=5, compute="bf16")

# Workload 4: small-M forward sweep on the same matrices.
W4 = dict(name="Llama-3-8B-shaped matrices, forward, M in {1,2,4,8,16}, r=8, alpha=16",
          shapes=LLAMA8B_LAYER, Ms=(1, 2, 4, 8, 16), r=8, alpha=16.0, compute="bf16")

# Workload 5: 1-D quantize/dequantize sweep.
W5 = dict(name="1-D NF4 double-quant sweep", sizes=tuple(2 ** e for e in (20, 22, 24, 26, 28, 30)) +
          (2 ** 20 + 7 * 16384,), std=0.02, outlier_frac=0.001, outlier_mult=50.0)

# Workload 6: selected rows of a Llama-3-8B-shaped NF4 embedding table.
W6 = dict(name="NF4 double-quant embedding 128256 x 4096, 4096 token ids, bf16 rows",
          rows=128256, dim=4096, n_ids=4096)

# Workload 7: merged deployment weight of the gate projection.
W7 = dict(name="merged fp32 weight of a 14336 x 4096 NF4 double-quant base, r=16, alpha=16",
          N=14336, K=4096, r=16, alpha=16.0)


def seed_for(workload: int, tensor_id: int) -> int:
    return BASE_SEED + 1000 * workload + tensor_id


def rng(workload: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(workload, tensor_id)))


def normal(shape, std, workload, tensor_id, dtype=np.float32) -> np.ndarray:
    return (rng(workload, tensor_id).standard_normal(shape) * std).astype(dtype)


def student_t(shape, df, scale, workload, tensor_id) -> np.ndarray:
    g = rng(workload, tensor_id)
    z0 = g.standard_normal(shape)
    chi2 = np.zeros(shape)
    for _ in range(df):
        chi2 += g.standard_normal(shape) ** 2
    return (z0 / np.sqrt(chi2 / df) * scale).astype(np.float32)


def with_outliers(x: np.ndarray, frac, mult, workload, tensor_id) -> np.ndarray:
    g = rng(workload, tensor_id)
    n = max(1, int(round(x.size * frac)))
    idx = g.choice(x.size, size=n, replace=False)
    y = x.copy().ravel()
    y[idx] *= mult
    return y.reshape(x.shape)


def adapters(N, K, r, workload, tensor_id):
    """LoRA factors: A ~ N(0, 1/r) [r, K], B ~ N(0, 0.01) [N, r] (B non-zero so dA is not vacuous)."""
    A = normal((r, K), 1.0 / r, workload, tensor_id)
    B = normal((N, r), 0.01, workload, tensor_id + 1)
    return A, B


def device_normal(shape, std, seed, device, dtype):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def device_student_t(shape, df, scale, seed, device, dtype):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z0 = torch.randn(shape, generator=g, device=device)
    chi2 = torch.zeros(shape, device=device)
    for _ in range(df):
        chi2 += torch.randn(shape, generator=g, device=device) ** 2
    return (z0 / torch.sqrt(chi2 / df) * scale).to(dtype)


def random_nf4_parts(n_packed, n_blocks, n_nested, double_quant, workload, tensor_id) -> dict:
    """Random stored bytes of an NF4 tensor, sized by the caller: any byte pattern is a
    valid stored tensor.  packed: uniform bytes; with double quantization absmax holds
    uniform uint8 codes, nested U(0.01, 0.05) float32 and offset 0.03; without it absmax
    is |N(0, 0.05)| + 0.001 float32."""
    g = rng(workload, tensor_id)
    packed = g.integers(0, 256, size=n_packed, dtype=np.uint8)
    if double_quant:
        return dict(packed=packed, absmax=g.integers(0, 256, size=n_blocks, dtype=np.uint8),
                    nested=g.uniform(0.01, 0.05, size=n_nested).astype(np.float32),
                    offset=np.float32(0.03))
    return dict(packed=packed, absmax=(np.abs(g.standard_normal(n_blocks)) * 0.05 + 0.001).astype(np.float32),
                nested=None, offset=None)


def token_ids(n, rows, workload, tensor_id, dtype=np.int64) -> np.ndarray:
    """n ids drawn uniformly from [0, rows)."""
    return rng(workload, tensor_id).integers(0, rows, size=n).astype(dtype)
