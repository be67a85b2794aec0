"""Floating-point storage formats, written from their format definitions.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

* bfloat16: 1 sign, 8 exponent, 7 mantissa bits; the upper half of an IEEE
  binary32. Conversion from fp32 rounds to nearest, ties to even (this is what
  ``tensor.to(torch.bfloat16)`` does in int4_per_token_head.py, reshape_and_cache_int4
  and unified_attention_int4, and what ``x.to(tl.bfloat16)`` does in kpool_compress.py,
  _fwht_quant_kernel).
* float16: IEEE binary16 (bias 15). The TurboQuant slot stores the value scale and
  zero as little-endian float16 words (triton_turboquant_decode.py, _tq_decode_stage1,
  value dequantize section).
* float8 E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities,
  S.1111.111 is NaN, largest finite 448 (the "e4nv" format that
  triton_turboquant_decode.py, _use_fp8_e4b15 selects on sm_89 and newer).
"""

import numpy as np

# ----------------------------------------------------------------------------
# bfloat16
# ----------------------------------------------------------------------------


def bf16_round(x):
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    The binary32 word is split into the kept upper 16 bits and the dropped lower
    16 bits. The kept part is incremented (in sign-magnitude, so a carry moves
    into the exponent and the largest finite value overflows to infinity) when
    the dropped part is more than half an ulp, or exactly half and the kept LSB
    is odd. NaNs stay NaN (quieted).
    """
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    kept = bits >> 16
    dropped = bits & 0xFFFF
    half = 0x8000
    round_up = (dropped > half) | ((dropped == half) & ((kept & 1) == 1))
    out = (kept + round_up.astype(np.uint64)) << 16
    nan = np.isnan(x)
    out = np.where(nan, ((bits >> 16) | 0x0040) << 16, out)
    return out.astype(np.uint32).view(np.float32).reshape(x.shape)


def bf16_bits(x):
    """bfloat16 bit patterns (uint16) of float32 values that are already bf16."""
    x = np.asarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(u16):
    """float32 values of bfloat16 bit patterns."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


# ----------------------------------------------------------------------------
# float16
# ----------------------------------------------------------------------------


def fp16_to_f64(u16):
    """Decode IEEE binary16 bit patterns to float64 from the format definition."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.int64)
    sign = np.where((u >> 15) & 1, -1.0, 1.0)
    e = (u >> 10) & 0x1F
    m = (u & 0x3FF).astype(np.float64)
    normal = sign * (1.0 + m / 1024.0) * np.exp2(e.astype(np.float64) - 15.0)
    subnormal = sign * (m / 1024.0) * np.exp2(-14.0)
    special = np.where(m == 0, sign * np.inf, np.nan)
    out = np.where(e == 0, subnormal, np.where(e == 31, special, normal))
    return out


# ----------------------------------------------------------------------------
# float8 E4M3FN
# ----------------------------------------------------------------------------


def e4m3fn_to_f64(u8):
    """Decode E4M3FN bytes to float64 from the format definition.

    exponent field e (4 bits, bias 7), mantissa field m (3 bits):
      e == 0            -> (-1)^s * m/8 * 2^-6        (subnormal)
      e == 15, m == 7   -> NaN                       (no infinities)
      otherwise         -> (-1)^s * (1 + m/8) * 2^(e-7)
    """
    u = np.asarray(u8, dtype=np.uint8).astype(np.int64)
    sign = np.where((u >> 7) & 1, -1.0, 1.0)
    e = (u >> 3) & 0xF
    m = (u & 0x7).astype(np.float64)
    normal = sign * (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = sign * (m / 8.0) * np.exp2(-6.0)
    out = np.where(e == 0, subnormal, normal)
    out = np.where((e == 15) & (m == 7), np.nan, out)
    return out


_E4M3_POS_VALUES = e4m3fn_to_f64(np.arange(0x7F, dtype=np.uint8))  # codes 0..126, increasing


def f32_to_e4m3fn(x):
    """Encode float32 values as E4M3FN bytes: nearest finite value, ties to even.

    Magnitudes beyond 448 saturate to 448 (the kernels only ever encode values that
    are clamped to [-448, 448] first, kpool_compress.py, _fwht_quant_kernel); NaN
    encodes as 0x7F. The sign bit is kept for zero.
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    vals = _E4M3_POS_VALUES
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_hi = np.abs(vals[hi] - a)
    d_lo = np.abs(a - vals[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((lo & 1) == 0))
    code = np.where(pick_lo, lo, hi)
    code = np.where(a >= 448.0, 0x7E, code)
    sign = (x.view(np.uint32) >> 31).astype(np.int64)
    out = (code | (sign << 7)).astype(np.uint8)
    out = np.where(np.isnan(x), np.uint8(0x7F), out)
    return out.astype(np.uint8)
