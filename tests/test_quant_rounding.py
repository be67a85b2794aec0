"""The write kernel's rounding shortcut against the oracle's definition (host check, no GPU).

int4_per_token_head.py, _reshape_cache_int4_kernel rounds half away from zero (where(u >= 0,
int(u + 0.5), int(u - 0.5)) in fp32) and clamps to [0, 15]. The kernel instead computes
w = saturate(fma(u, 2^-4, 2^-5)) -- fl(u + 0.5) / 16, since the product is exact and the fused
add rounds once -- then adds 2^19 under round-toward-zero (the ulp at 2^19 is 2^-4, so the low
bits hold trunc(16 w)) and takes an integer min with 15. These tests run that formula in numpy over
every fp32 u in [0.25, 17) (where the rounding of u + 0.5 and the clamp matter), random values
elsewhere and the special values, against oracle.int4_cache.round_half_away."""

import numpy as np

from oracle import int4_cache

F32 = np.float32


def _kernel_formula(u):
    u = np.asarray(u, dtype=F32)
    with np.errstate(invalid="ignore", over="ignore"):
        # fma(u, 1/16, 1/32): the exact value rounded once to fp32 (float64 holds u/16 + 1/32 exactly
        # wherever the result is not simply 1/32)
        w = (u.astype(np.float64) * 0.0625 + 0.03125).astype(F32)
        w = np.where(np.isnan(w), F32(0.0), np.clip(w, F32(0.0), F32(1.0)))  # .sat: NaN -> 0
    # w + 2^19 with round-toward-zero lands on the grid of step 2^-4: the field above 2^19 is trunc(16 w)
    field = np.floor((w.astype(np.float64) + 524288.0) * 16.0) - 8388608.0
    return np.minimum(field, 15.0).astype(np.int64)


def _oracle(u):
    q = int4_cache.round_half_away(np.asarray(u, dtype=F32)).astype(np.float64)
    return np.clip(q, 0, 15).astype(np.int64)


def test_every_fp32_value_where_rounding_matters():
    # every fp32 in [0.25, 17): the half-integers, the rounding of u + 0.5 near 1, and the clamp
    lo, hi = np.float32(0.25).view(np.uint32), np.float32(17.0).view(np.uint32)
    for start in range(int(lo), int(hi), 1 << 22):
        u = np.arange(start, min(start + (1 << 22), int(hi)), dtype=np.uint32).view(F32)
        assert np.array_equal(_kernel_formula(u), _oracle(u))


def test_sampled_fp32_values_elsewhere():
    # below 0.25 (u + 0.5 < 1, both give 0) and below 0: random bit patterns
    rng = np.random.default_rng(7)
    tiny = rng.integers(0, np.float32(0.25).view(np.uint32), size=1 << 20, dtype=np.uint32).view(F32)
    neg = -rng.integers(0, np.float32(3e38).view(np.uint32), size=1 << 20, dtype=np.uint32).view(F32)
    big = rng.integers(np.float32(17.0).view(np.uint32), np.float32(3e38).view(np.uint32), size=1 << 20,
                       dtype=np.uint32).view(F32)
    for u in (tiny, neg, big):
        assert np.array_equal(_kernel_formula(u), _oracle(u))


def test_special_values():
    u = np.array([np.nan, np.inf, -np.inf, 1e30, -1e30, 3.4e38, -3.4e38, 0.49999997, 0.5, 14.5,
                  15.4999990, 15.5, 16.0, 1e7, -1e7, -0.0], dtype=F32)
    assert np.array_equal(_kernel_formula(u), _oracle(u))
    # the pages' fp32 add makes 0.49999997 round up to 1 (not 0): both sides keep it
    assert _oracle(np.array([0.49999997], dtype=F32))[0] == 1
