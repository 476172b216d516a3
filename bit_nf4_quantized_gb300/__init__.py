"""NF4 double-quantized frozen-base QLoRA linear for one NVIDIA GB300 (sm_103a).

The computation lives in ``libqlora_nf4.so`` (CUDA kernels behind the C ABI of
``include/qlora_nf4.h``); :mod:`.binding` is the ctypes layer that marshals PyTorch
tensors to it.  Build the library with ``python -m bit_nf4_quantized_gb300.build``.
"""

from .binding import (Nf4Error, Nf4Tensor, code_tables, device_status, launch_count,  # noqa: F401
                      nf4_dequantize, nf4_embedding_rows, nf4_merge_lora, nf4_quantize,
                      qlora_linear_bwd, qlora_linear_fwd)
