"""Plain CPU oracle for NF4 double quantization and the frozen-base QLoRA linear.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or link
anything in this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares no
code, tables or constant generators with the CUDA library in
``bit_nf4_quantized_gb300/csrc``; the two are tied together only by tests that
compare their outputs on the same seeded inputs.

Sources (the web pages this work follows):
  [ADAPT] "Native model adaptation and NF4" (anerlang.org/docs/gen-adaptation),
          section "Packed NF4 and the portable QLoRA profile" -- the storage format;
          section "Adapter API" / "LoRA FA includes gradient preconditioning" --
          rank bounds and s = alpha / rank;
          section "Fused GPU NF4 decodes inside the matrix kernel" -- decode semantics.
  [GATE]  "NF4 Layer Streaming -- Gate results" (Soup, benchmarks/gate-v0.72.2-nf4.md),
          section "P3 is solved, and the probe that settles it" -- bytes per
          parameter, shared constant code tables, deterministic requantization.
  [QUAL]  V100 accelerated qualification record
          (native_training_accelerated_20261031.json), keys ``component_benchmarks``
          (packed GPU bytes per matrix) and ``jit.kernel_identity`` (separately
          rounded decode, no atomics).
  [QUAL-2] CPU/V100 adaptation record (native_adaptation_20261030.json), key
          ``nf4`` (block 64, nested block 256, dynamic8) and the ``nf4_base.memory``
          byte totals.

Modules: ``codebooks`` (the two code tables), ``nf4`` (quantize / dequantize /
byte formula), ``qlora`` (linear forward and backward in float64), ``export``
(selected embedding rows, merged LoRA weight).  Every
function is pinned by ``tests/test_oracle_*.py`` against facts the pages or the
mathematics fix; see each module header.
"""

from . import codebooks, export, nf4, qlora  # noqa: F401
