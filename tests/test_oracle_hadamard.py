"""Pins for oracle/hadamard.py: textbook closed form, exact integer products, inverse identity."""

import numpy as np
import pytest

from oracle import hadamard


def _closed_form(d):
    """Sylvester Hadamard entries: H[i, j] = (-1)^popcount(i & j)."""
    i = np.arange(d)[:, None]
    j = np.arange(d)[None, :]
    x = i & j
    pc = np.zeros_like(x)
    while np.any(x):
        pc += x & 1
        x >>= 1
    return np.where(pc % 2 == 0, 1, -1)


@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_sylvester_closed_form_and_orthogonality(d):
    H = hadamard.sylvester(d)
    assert np.array_equal(H, _closed_form(d))
    assert np.array_equal(H, H.T)
    assert np.array_equal(H @ H.T, d * np.eye(d, dtype=np.int64))


@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128, 256])
def test_butterfly_equals_matrix_on_integers(d):
    rng = np.random.default_rng(d)
    x = rng.integers(-100, 101, size=(7, d))
    H = _closed_form(d)
    exact = x @ H.T
    assert np.array_equal(hadamard.fwht(x.astype(np.float32)), exact.astype(np.float32))
    assert np.array_equal(hadamard.fwht(x.astype(np.float64)), exact.astype(np.float64))
    # H_d H_d = d I: applying the unnormalised transform twice scales by d
    assert np.array_equal(hadamard.fwht(hadamard.fwht(x.astype(np.float64))), d * x)


def test_butterfly_fp32_within_rounding_bound():
    rng = np.random.default_rng(5)
    for d in (64, 128):
        x = rng.standard_normal((500, d)).astype(np.float32)
        got = hadamard.fwht(x).astype(np.float64)
        exact = x.astype(np.float64) @ _closed_form(d).T
        # log2(d) additions, each adding at most half an ulp of a partial sum bounded by sum|x|
        bound = np.log2(d) * np.abs(x).astype(np.float64).sum(axis=1, keepdims=True) * 2.0**-24
        assert np.all(np.abs(got - exact) <= bound)


def test_rht_inverse_identity():
    rng = np.random.default_rng(6)
    d = 128
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    x = rng.integers(-50, 51, size=(4, d)).astype(np.float32)
    y = hadamard.rht_forward(x, signs)
    assert np.array_equal(hadamard.rht_inverse_f64(y, signs), d * x.astype(np.float64))


def test_normalised_h128_is_orthonormal():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((300, 128)).astype(np.float32)
    y = hadamard.hadamard128_normalised_f32(x).astype(np.float64)
    exact = x.astype(np.float64) @ _closed_form(128).T / np.sqrt(128.0)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x.astype(np.float64), axis=1), rtol=1e-6)
    assert np.max(np.abs(y - exact)) < 1e-4
    assert hadamard.H128_SCALE_F32 == np.float32(1.0 / np.sqrt(128.0))
