"""Pins for oracle/formats.py: each conversion against a library routine and the format definition."""

import numpy as np
import torch

from oracle import formats


def _special_f32():
    vals = [0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, np.inf, -np.inf, 1e-40, -1e-40, 1.17549435e-38]
    bits = [0x7F7FFFFF, 0xFF7FFFFF, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001,
            0x00008000, 0x00018000, 0x7F7F8000, 0x7F7F7FFF, 0x7F7E8000]
    a = np.array(vals, dtype=np.float32)
    b = np.array(bits, dtype=np.uint32).view(np.float32)
    return np.concatenate([a, b])


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(30.0),
        rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32),
        _special_f32(),
    ])
    x = x[~np.isnan(x)]
    mine = formats.bf16_bits(formats.bf16_round(x))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_round_ties_to_even_by_hand():
    # 1 + 2^-8 is exactly halfway between bf16 1.0 and 1.0078125: even mantissa -> 1.0
    assert formats.bf16_round(np.float32(1.0 + 2.0**-8)) == np.float32(1.0)
    # 1.0078125 + 2^-8 is halfway between 1.0078125 (odd) and 1.015625 (even) -> up
    assert formats.bf16_round(np.float32(1.0078125 + 2.0**-8)) == np.float32(1.015625)
    assert np.isnan(formats.bf16_round(np.float32(np.nan)))
    assert formats.bf16_round(np.float32(3.4e38)) == np.inf


def test_fp16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    mine = formats.fp16_to_f64(codes)
    ref = codes.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = formats.e4m3fn_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    # spot values from the format definition (bias 7, 3 mantissa bits, S.1111.111 = NaN)
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x01] == 2.0**-9 and mine[0x08] == 2.0**-6 and mine[0x38] == 1.0
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    assert np.sum(np.isnan(mine)) == 2


def test_e4m3_encode_round_trip_and_ties():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = formats.e4m3fn_to_f64(codes).astype(np.float32)
    assert np.array_equal(formats.f32_to_e4m3fn(vals), codes)
    pos = formats.e4m3fn_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # midpoints exact in fp32
    enc = formats.f32_to_e4m3fn(mids).astype(np.int64)
    lo = np.arange(0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(enc, expect)


def test_e4m3_encode_brute_force_and_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-448, 448, 100000),
        rng.standard_normal(100000) * 4,
        rng.standard_normal(50000) * 1e-2,
    ]).astype(np.float32)
    enc = formats.f32_to_e4m3fn(x)
    got = formats.e4m3fn_to_f64(enc)
    finite = formats.e4m3fn_to_f64(np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8))
    best = np.min(np.abs(finite[None, :] - x[:5000, None].astype(np.float64)), axis=1)
    assert np.array_equal(np.abs(got[:5000] - x[:5000]), best)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch keeps the sign of zero results too; compare values (and bytes away from zero)
    assert np.array_equal(formats.e4m3fn_to_f64(ref), got)
