"""Fused normalised FWHT-128 + per-row power-of-two absmax FP8 quantizer.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source page: kpool_compress.py, _fwht_quant_kernel / fwht128_quant_fp8. Per row
of 128 bf16 values, in fp32:
  1. x = 7 butterfly stages (stride 1..64) * 0.08838834764831845  (_hadamard128);
  2. x = bf16(x) (the unfused path's bf16 materialisation);
  3. a = max(max |x|, 1e-4);
  4. s = 2^ceil(log2(a * (1/448)))  -- read as exact math: the smallest power of
     two that is >= the fp32 product a * fp32(1/448);
  5. y = clamp(x / s, -448, 448), stored as FP8 E4M3FN (round to nearest even);
outputs y [rows, 128] (E4M3FN bytes) and s [rows] (fp32).
"""

import numpy as np

from .formats import bf16_round, f32_to_e4m3fn
from .hadamard import hadamard128_normalised_f32

F32 = np.float32


def pow2_ceil(m):
    """Smallest power of two >= m for positive finite float32 m (exact)."""
    m = np.asarray(m, dtype=np.float32)
    frac, exp = np.frexp(m.astype(np.float64))         # m = frac * 2^exp, frac in [0.5, 1)
    p = np.where(frac == 0.5, exp - 1, exp)
    return np.ldexp(np.float64(1.0), p).astype(np.float32)


def fwht128_quant_fp8(x):
    """x: [rows, 128] float32 holding bf16 values -> (codes uint8 [rows, 128], scale float32 [rows])."""
    x = np.asarray(x, dtype=np.float32)
    assert x.ndim == 2 and x.shape[1] == 128
    y = bf16_round(hadamard128_normalised_f32(x))
    a = np.maximum(np.abs(y).max(axis=1), F32(1e-4)) if y.shape[0] else np.zeros((0,), F32)
    m = (a * F32(1.0 / 448.0)).astype(np.float32)
    s = pow2_ceil(m) if y.shape[0] else np.zeros((0,), F32)
    q = np.clip(y / s[:, None], F32(-448.0), F32(448.0)).astype(np.float32)
    return f32_to_e4m3fn(q), s.astype(np.float32)
