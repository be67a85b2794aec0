"""Walsh-Hadamard transforms.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: int4_per_token_head.py, section "Randomized Hadamard Transform (RHT)":
  * _get_hadamard_matrix builds the Sylvester matrix by the doubling
    H_2n = [[H_n, H_n], [H_n, -H_n]] starting from [[1]];
  * fast_hadamard_transform is the unnormalised transform H_d x with
    H_d H_d = d I; its PyTorch tier is a butterfly whose stage h (h = 1, 2, 4, ...)
    views the last axis as blocks of 2h, and inside each block replaces the pair
    (a, b) = (x[j], x[h + j]) by (a + b, a - b);
  * single_rht applies H(x * d1) forward and H(x) * d1 backward (signs d1 = +-1).
Source: kpool_compress.py, _hadamard128 / _fwht_quant_kernel: the same seven
butterfly stages (stride 1, 2, ..., 64) on 128 lanes, then one fp32 multiply by
0.08838834764831845 (1/sqrt(128) rounded to fp32).

The butterfly here works in the dtype of its input (float32 -> every add and
subtract is rounded to fp32, exactly like the pages' fp32 tensors).
"""

import numpy as np


def sylvester(d):
    """The d x d Sylvester Hadamard matrix (int64), by repeated doubling."""
    assert d >= 1 and d & (d - 1) == 0, d
    H = np.ones((1, 1), dtype=np.int64)
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def fwht(x):
    """Unnormalised WHT along the last axis by the butterfly; keeps x's dtype.

    Stage h takes each block of 2h elements, splits it into the first half a and
    the second half b, and writes (a + b, a - b).
    """
    x = np.array(x, copy=True)
    d = x.shape[-1]
    assert d & (d - 1) == 0, d
    h = 1
    while h < d:
        blocks = x.reshape(x.shape[:-1] + (d // (2 * h), 2, h))
        a = blocks[..., 0, :]
        b = blocks[..., 1, :]
        x = np.stack([a + b, a - b], axis=-2).reshape(x.shape)
        h *= 2
    return x


def rht_forward(x_f32, signs):
    """H (x * d1) in fp32 (int4_per_token_head.py, single_rht, forward)."""
    x = np.asarray(x_f32, dtype=np.float32)
    return fwht(x * np.asarray(signs, dtype=np.float32))


def rht_inverse_f64(y, signs):
    """H(y) * d1 in float64 (int4_per_token_head.py, single_rht, inverse=True)."""
    y = np.asarray(y, dtype=np.float64)
    return fwht(y) * np.asarray(signs, dtype=np.float64)


H128_SCALE_F32 = np.float32(0.08838834764831845)  # 1/sqrt(128) rounded to fp32


def hadamard128_normalised_f32(x_f32):
    """kpool_compress.py, _hadamard128: seven fp32 butterfly stages, then * 1/sqrt(128)."""
    x = np.asarray(x_f32, dtype=np.float32)
    assert x.shape[-1] == 128
    return fwht(x) * H128_SCALE_F32
