"""Reference oracle for the quantized paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, CPU implementation
written from the source pages (int4_per_token_head.py, triton_turboquant_decode.py,
kpool_compress.py). It exists to check the CUDA library, never to stand in for
it: only the test suite, the smoke check and the benchmark's CPU-baseline leg
may import it. It shares no code with the CUDA path and imports nothing from it.

Precision: the INT4 quantizer and the FWHT-128/FP8 codec run in IEEE fp32 with
the pages' operation order (the pages fix that precision: Triton fp32 kernels);
attention runs in float64.

Modules
  formats      bf16 / fp16 / FP8-E4M3FN conversions from their format definitions
  hadamard     Sylvester Hadamard matrix and the fp32 butterfly FWHT
  int4_cache   RHT + INT4 quantize + nibble pack + page scatter, dequant, decode
  turboquant   decode over the FP8-key / 3-4-bit-value combined slot layout
  fwht_fp8     fused normalised FWHT-128 + power-of-two absmax FP8 quantizer
  kpool        pooled softmax-weighted key -> Hadamard-128 -> FP8 -> paged write (kpool_compress.py)

Every function is pinned by tests that do not re-use it (see tests/test_oracle_*.py).
"""

from . import formats, hadamard, int4_cache, turboquant, fwht_fp8, kpool  # noqa: F401
