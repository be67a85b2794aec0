"""kvq_decode_tq_mse (TurboQuant, MSE keys) on the GPU against the float64 oracle on the same
cache bytes, rotation and codebook. Tolerance: 2e-3 + 1e-2 |oracle| elementwise."""

import numpy as np
import pytest
import torch

from oracle import turboquant
from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import MseCase, assert_close, scatter_into_pool

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("key_bits,value_bits", [(3, 4), (4, 4), (3, 3), (4, 3)])
@pytest.mark.parametrize("Hk,G,D", [(8, 4, 128), (2, 2, 64), (1, 8, 128), (16, 1, 64)])
def test_small_layouts(key_bits, value_bits, Hk, G, D):
    lens = [1, 15, 16, 17, 100, 0, 40]
    case = workloads.DecodeCase("mse", len(lens), Hk * G, Hk, D, lens, seed=key_bits * 10 + value_bits + Hk + G)
    c = MseCase(case, key_bits, value_bits, num_blocks=sum(workloads.pages_needed(lens)) + 3)
    for corr in (False, True):
        ref = c.oracle(corr)
        for S in (0, 3):
            got = c.gpu(corr, S)
            assert_close(got, ref, what="k%d v%d Hk=%d G=%d D=%d corr=%d S=%d" % (key_bits, value_bits, Hk, G, D,
                                                                                 corr, S))
            assert np.all(got[5] == 0.0)


def test_padded_key_part():
    """key_packed_size past MSE_BYTES + 2 (values further into the slot, other byte alignment)."""
    lens = [33, 70]
    case = workloads.DecodeCase("pad", 2, 8, 2, 128, lens, seed=41)
    for pad in (2, 6, 14):
        c = MseCase(case, 3, 4, kps_pad=pad)
        assert_close(c.gpu(True), c.oracle(True), what="pad %d" % pad)


@pytest.mark.parametrize("key_bits,value_bits", [(3, 4), (4, 3)])
def test_full_size_sampled(key_bits, value_bits):
    """B=64, Hq=32, Hk=8, D=128, seq_len 4096: the benchmark's launch; oracle on sampled sequences."""
    case = workloads.turboquant_mse(key_bits, value_bits)
    c = MseCase(case, key_bits, value_bits)
    got = c.gpu(False)
    idx = [0, 31, 63]
    assert_close(got[idx], c.oracle(False, batch_index=idx)[idx], what="mse full k%d v%d" % (key_bits, value_bits))


def test_pages_scattered_in_a_large_pool():
    """MSE-key slots scattered over a 200000-block pool (3.3 GB of 128-byte slots), its first and
    last blocks in use; the oracle reads the same pages compactly."""
    lens = [640, 33, 1500]
    case = workloads.DecodeCase("msepool", len(lens), 32, 8, 128, lens, seed=72)
    c = MseCase(case, 3, 4)
    pool, bt = scatter_into_pool(c.cache, c.bt, 200000, 72)
    out = kvq.kvq_decode_tq_mse(c.q.cuda(), c.Pi.cuda(), c.cb.cuda(), pool, c.kb, c.kps, c.vb, bt.cuda(),
                                c.lens.cuda(), c.scale)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0
    assert_close(out.cpu().numpy(), c.oracle(False), what="mse large pool")
    del pool
    torch.cuda.empty_cache()


def test_used_bytes_an_odd_multiple_of_16():
    """3-bit keys and values with the key part padded by 10: the used bytes of a slot are 112, an odd
    multiple of 16 (the staged row keeps 4 bytes past them for the unaligned read of the scale
    word, so the row is 144 wide)."""
    lens = [300, 47]
    case = workloads.DecodeCase("mse112", len(lens), 8, 2, 128, lens, seed=47)
    c = MseCase(case, 3, 3, kps_pad=10)
    assert c.kps + 48 + 4 == 112
    for corr in (False, True):
        assert_close(c.gpu(corr), c.oracle(corr), what="used 112 corr=%d" % corr)
