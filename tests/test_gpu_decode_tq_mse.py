"""kvq_decode_tq_mse (TurboQuant, MSE keys) on the GPU against the float64 oracle on the same
cache bytes, rotation and codebook. Tolerance: 2e-3 + 1e-2 |oracle| elementwise."""

import numpy as np
import pytest
import torch

from oracle import turboquant
from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import assert_close

pytestmark = pytest.mark.gpu


class MseCase:
    def __init__(self, case, key_bits, value_bits, num_blocks=None, kps_pad=0):
        self.case, self.kb, self.vb = case, key_bits, value_bits
        D, Hk = case.D, case.Hk
        mse, kps, sb = workloads.turboquant_mse_layout(D, key_bits, value_bits)
        if kps_pad:  # a larger key_packed_size (padding after the norm)
            kps += kps_pad
            sb = -(-(kps + (-(-D * value_bits // 8)) + 4) // 16) * 16
        self.kps, self.sb = kps, sb
        self.bt, self.nb = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=num_blocks)
        base = workloads.random_turboquant_mse_slots((self.nb, 16, Hk), D, key_bits, value_bits, case.seed)
        if kps_pad:  # move the value fields behind the padded key part
            m0, k0, s0 = workloads.turboquant_mse_layout(D, key_bits, value_bits)
            cache = torch.zeros((self.nb, 16, Hk, sb), dtype=torch.uint8)
            cache[..., :k0] = base[..., :k0]
            vlen = -(-D * value_bits // 8) + 4
            cache[..., kps:kps + vlen] = base[..., k0:k0 + vlen]
            base = cache
        self.cache = base
        self.q = workloads.query(case, dtype=torch.float32)
        self.Pi = workloads.random_rotation(D, case.seed)
        self.cb = workloads.mse_codebook(key_bits, D)
        self.lens = torch.tensor(case.seq_lens, dtype=torch.int32)
        self.scale = 1.0 / np.sqrt(D)

    def gpu(self, norm_correction, num_splits=0):
        out = kvq.kvq_decode_tq_mse(self.q.cuda(), self.Pi.cuda(), self.cb.cuda(), self.cache.cuda(), self.kb,
                                    self.kps, self.vb, self.bt.cuda(), self.lens.cuda(), self.scale,
                                    norm_correction=norm_correction, num_splits=num_splits)
        st, flags = kvq.kvq_device_error()
        assert st == 0 and flags == 0, (st, flags)
        return out.cpu().numpy()

    def oracle(self, norm_correction, batch_index=None):
        return turboquant.decode_tq_mse(self.q.numpy(), self.cache.numpy(), self.kb, self.kps, self.vb,
                                        self.cb.numpy(), norm_correction, self.Pi.numpy(), self.bt.numpy(),
                                        np.asarray(self.case.seq_lens), self.scale, batch_index=batch_index)


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
