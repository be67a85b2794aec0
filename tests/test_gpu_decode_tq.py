"""kvq_decode_tq (FP8 keys, 4-bit / 3-bit values) on the GPU against the float64 oracle."""

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import TqCase, assert_close, scatter_into_pool

pytestmark = pytest.mark.gpu


def _run(c, num_splits=0):
    out = kvq.kvq_decode_tq(c.q.cuda(), c.cache.cuda(), c.bits, c.bt.cuda(), c.lens.cuda(), c.scale,
                            num_splits=num_splits)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("Hk,G,D", [(8, 4, 128), (2, 2, 64), (1, 8, 128), (16, 1, 64)])
def test_small_layouts(bits, Hk, G, D):
    lens = [1, 16, 37, 300, 0, 129]
    case = workloads.DecodeCase("tq", len(lens), Hk * G, Hk, D, lens, seed=bits + Hk + G)
    c = TqCase(case, bits, num_blocks=sum(workloads.pages_needed(lens)) + 3)
    ref = c.oracle()
    for S in (0, 4):
        got = _run(c, S)
        assert_close(got, ref, what="bits=%d Hk=%d G=%d D=%d S=%d" % (bits, Hk, G, D, S))
        assert np.all(got[4] == 0.0)


@pytest.mark.parametrize("bits", [4, 3])
def test_turboquant_full_size_sampled(bits):
    """B=64, Hq=32, Hk=8, D=128, seq_len 4096: the full workload, oracle on sampled sequences."""
    c = TqCase(workloads.turboquant_fp8(bits), bits)
    got = _run(c)
    idx = [0, 40, 63]
    ref = c.oracle(batch_index=idx)
    assert_close(got[idx], ref[idx], what="tq full bits=%d" % bits)


@pytest.mark.parametrize("bits", [4, 3])
def test_slot_wider_than_its_fields(bits):
    """slot_bytes 48 past the key, values, scale and zero (zero padding that is never read): the
    page tiles take only each slot's used bytes."""
    lens = [5, 200, 33]
    case = workloads.DecodeCase("tqpad", len(lens), 16, 4, 128, lens, seed=90 + bits)
    c = TqCase(case, bits, num_blocks=sum(workloads.pages_needed(lens)) + 2)
    pad = torch.full(c.cache.shape[:-1] + (48,), 0xAB, dtype=torch.uint8)
    c.cache = torch.cat([c.cache, pad], dim=-1).contiguous()
    assert c.cache.shape[-1] % 16 == 0
    assert_close(_run(c), c.oracle(), what="padded slot bits=%d" % bits)


def test_pages_scattered_in_a_4gb_pool():
    """Pages scattered over a 150000-block pool (4 GB of 208-byte slots), its last block in use: the
    page tiles' tensor map addresses the whole pool. The oracle reads the same pages compactly."""
    lens = [300, 1000, 17]
    case = workloads.DecodeCase("tqpool", len(lens), 32, 8, 128, lens, seed=71)
    c = TqCase(case, 4)
    pool, bt = scatter_into_pool(c.cache, c.bt, 150000, 71)
    out = kvq.kvq_decode_tq(c.q.cuda(), pool, 4, bt.cuda(), c.lens.cuda(), c.scale)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0
    assert_close(out.cpu().numpy(), c.oracle(), what="tq 4 GB pool")
    del pool
    torch.cuda.empty_cache()
