"""kvq_kpool_write on the GPU against the oracle (oracle/kpool.py): every cache byte bit-exact --
the FP8 codes, the fp32 scales, and the bytes that must stay untouched."""

import numpy as np
import pytest
import torch

from oracle import kpool
from quantized_paged_kv_int4_gb300 import kvq, workloads

pytestmark = pytest.mark.gpu


def _both(n, pool, ps, seed, round_scale=True, mask=None, loc_override=None):
    slot_k, score, ape, loc, nb = workloads.kpool_case(n, pool, ps, seed)
    if loc_override is not None:
        loc = loc_override
    cache = np.full((nb, ps, 132), 0x5A, np.uint8)
    ref = cache.copy()
    m = None if mask is None else mask.numpy()
    ok = (loc >= 0) & (loc < nb * ps)
    if m is not None:
        m = m & ok.numpy()
    elif not bool(ok.all()):
        m = ok.numpy()
    kpool.kpool_compress_write(ref, slot_k.float().numpy(), score.numpy(), ape.numpy(), loc.numpy(), m, round_scale)
    g = torch.from_numpy(cache).cuda()
    kvq.kvq_kpool_write(g, slot_k.cuda(), score.cuda(), ape.cuda(), loc.cuda(),
                        None if mask is None else mask.cuda(), round_scale=round_scale)
    st, flags = kvq.kvq_device_error()
    return g.cpu().numpy(), ref, st, flags


@pytest.mark.parametrize("pool", [1, 4, 7, 16])
@pytest.mark.parametrize("round_scale", [True, False])
def test_bit_exact(pool, round_scale):
    got, ref, st, flags = _both(333, pool, 16, seed=pool, round_scale=round_scale)
    assert st == 0 and flags == 0
    assert np.array_equal(got, ref)


def test_write_mask_and_page_size_64():
    n = 1000
    mask = torch.rand((n,), generator=torch.Generator().manual_seed(5)) < 0.7
    got, ref, st, flags = _both(n, 4, 64, seed=9, mask=mask)
    assert st == 0 and flags == 0
    assert np.array_equal(got, ref)


def test_out_of_range_location_is_skipped_and_flagged():
    n = 40
    _, _, _, loc, nb = workloads.kpool_case(n, 4, 16, 11)
    loc = loc.clone()
    loc[3] = nb * 16          # one past the pool
    loc[17] = -5
    got, ref, st, flags = _both(n, 4, 16, seed=11, loc_override=loc)
    assert st != 0 and flags != 0
    assert np.array_equal(got, ref)


def test_full_size_16384_pools():
    """16384 pools of 4 tokens (65536 tokens), pages of 64: the benchmark's launch."""
    got, ref, st, flags = _both(16384, 4, 64, seed=0)
    assert st == 0 and flags == 0
    assert np.array_equal(got, ref)
