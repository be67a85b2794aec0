"""kvq_fwht128 on the GPU against the oracle: E4M3 codes and power-of-two scales bit-exact."""

import numpy as np
import pytest
import torch

from oracle import fwht_fp8
from quantized_paged_kv_int4_gb300 import kvq, workloads

pytestmark = pytest.mark.gpu


def _check(x):
    y, s = kvq.kvq_fwht128(x.cuda())
    codes, scale = fwht_fp8.fwht128_quant_fp8(workloads.to_numpy_f32(x))
    assert np.array_equal(y.view(torch.uint8).cpu().numpy(), codes)
    assert np.array_equal(s.cpu().numpy()[:, 0], scale)


def test_full_size_65536_rows():
    _check(workloads.fwht_rows(65536))


@pytest.mark.parametrize("rows", [1, 15, 17, 33])
def test_ragged_row_counts(rows):
    _check(workloads.fwht_rows(rows, seed=rows))


def test_special_rows():
    x = workloads.fwht_rows(64, seed=5).float()
    x[0] = 0.0                                   # absmax floor 1e-4
    x[1] = 0.0
    x[1, 0] = 1.0                                # e_0: every output 362 / 2^12 -> 352
    x[2] *= 1e-30                                # tiny: subnormal E4M3 outputs
    x[3] *= 1e30                                 # huge but finite
    x[4] = torch.linspace(-3, 3, 128)
    x[5, ::2] = 448.0                            # exactly representable pattern
    x[6] = -x[6].abs()
    _check(x.to(torch.bfloat16))


def test_empty():
    y, s = kvq.kvq_fwht128(torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"))
    assert y.shape == (0, 128) and s.shape == (0, 1)
