"""Pins for oracle/fwht_fp8.py (kpool_compress.py, _fwht_quant_kernel)."""

import numpy as np
import torch

from oracle import formats, fwht_fp8, hadamard


def test_worked_example_unit_vector():
    # e_0 -> all ones after the unnormalised transform; * fp32(1/sqrt 128) = 0.0883883461..
    # -> bf16 0x3DB5 = 0.08837890625; absmax * fp32(1/448) = 1.9727e-4 lies in (2^-13, 2^-12]
    # -> scale 2^-12; 0.08837890625 * 4096 = 362 -> nearest E4M3 is 352 (1.011b * 2^8) = 0x7B.
    x = np.zeros((2, 128), np.float32)
    x[0, 0] = 1.0
    x[1, 0] = -1.0
    codes, scale = fwht_fp8.fwht128_quant_fp8(x)
    assert np.all(codes[0] == 0x7B) and np.all(codes[1] == 0xFB)
    assert np.all(scale == np.float32(2.0**-12))
    assert formats.bf16_round(hadamard.H128_SCALE_F32) == np.float32(0.08837890625)


def test_zero_row_uses_floor():
    # absmax floor 1e-4: 1e-4 * fp32(1/448) = 2.23e-7 in (2^-23, 2^-22] -> scale 2^-22, codes 0
    codes, scale = fwht_fp8.fwht128_quant_fp8(np.zeros((1, 128), np.float32))
    assert np.all(codes == 0) and scale[0] == np.float32(2.0**-22)


def test_pow2_ceil_closed_forms():
    for k in (-30, -12, -1, 0, 5, 100):
        p = np.float32(2.0**k)
        assert fwht_fp8.pow2_ceil(p) == p
        assert fwht_fp8.pow2_ceil(np.float32(p * np.float32(1 + 2**-23))) == np.float32(2.0 ** (k + 1))
        assert fwht_fp8.pow2_ceil(np.float32(0.75 * 2.0**k)) == p


def test_invariants_on_random_rows():
    rng = np.random.default_rng(3)
    x = formats.bf16_round((rng.standard_normal((3000, 128)) * rng.uniform(1e-3, 1e3, (3000, 1))).astype(np.float32))
    codes, s = fwht_fp8.fwht128_quant_fp8(x)
    frac, _ = np.frexp(s.astype(np.float64))
    assert np.all(frac == 0.5)                                   # powers of two
    y = formats.bf16_round(hadamard.hadamard128_normalised_f32(x))
    a = np.maximum(np.abs(y).max(1), np.float32(1e-4)).astype(np.float64)
    ratio = a / s
    assert np.all((ratio > 224 * (1 - 2**-22)) & (ratio <= 448 * (1 + 2**-22)))
    # the quantization step against torch's own fp32 -> float8_e4m3fn cast
    scaled = np.clip(y / s[:, None], -448, 448).astype(np.float32)
    ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(formats.e4m3fn_to_f64(codes), ref)
    # end to end against the exact transform: within one E4M3 half-step plus bf16 rounding
    exact = x.astype(np.float64) @ hadamard.sylvester(128).T / np.sqrt(128.0)
    deq = formats.e4m3fn_to_f64(codes) * s[:, None]
    tol = np.abs(exact) * (2.0**-4 + 2.0**-8) + s[:, None] * 2.0**-9 + 1e-6 * np.abs(exact).max(1, keepdims=True)
    assert np.all(np.abs(deq - exact) <= tol)
