"""Shared builders for the GPU parity tests: seeded inputs (workloads), the oracle's result on
the CPU, and the same inputs uploaded to the GPU. Nothing here reads data back from the CUDA
path into an oracle input."""

import math

import numpy as np
import torch

from oracle import int4_cache, turboquant
from quantized_paged_kv_int4_gb300 import workloads

# attention output tolerance (elementwise): |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL = 2e-3
RTOL = 1e-2


def assert_close(gpu, ref, atol=ATOL, rtol=RTOL, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), "%s: %d/%d outside tolerance, max err %.3e at %s" % (
        what, int(bad.sum()), bad.size, err.max(), np.unravel_index(np.argmax(err), err.shape))
    return float(err.max())


class Int4Case:
    """An INT4 decode case whose cache the ORACLE wrote (from seeded K / V), or random bytes."""

    def __init__(self, case, signs=True, num_blocks=None, random_cache=False, scale_mult=1.0,
                 unused_fill=0, kv_transform=None):
        self.case = case
        D, Hk = case.D, case.Hk
        self.bt, self.nb = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=num_blocks,
                                                  unused_fill=unused_fill)
        self.signs = workloads.rht_signs(D) if signs else None
        self.scale = scale_mult / math.sqrt(D)
        nb = self.nb
        if random_cache:
            kb, vb, kw, vw = workloads.random_int4_pages(nb, Hk, D, case.seed)
            self.kc, self.vc = kb.numpy(), vb.numpy()
            self.ks = kw.numpy().view(np.uint32)
            self.vs = vw.numpy().view(np.uint32)
        else:
            _, _, slots = workloads.all_token_slots(self.bt, case.seq_lens)
            k, v = workloads.kv_vectors(case, slots.numel())
            if kv_transform is not None:  # (k, v) bf16 [T, Hk, D] -> (k, v) before the write
                k, v = kv_transform(k, v)
            self.kc = np.zeros((nb, 16, Hk, D // 2), np.uint8)
            self.vc = np.zeros_like(self.kc)
            self.ks = np.zeros((nb, 16, Hk), np.uint32)
            self.vs = np.zeros_like(self.ks)
            int4_cache.write_int4(workloads.to_numpy_f32(k), workloads.to_numpy_f32(v), slots.numpy(),
                                  None if self.signs is None else self.signs.numpy(),
                                  self.kc, self.vc, self.ks, self.vs)
        self.q = workloads.query(case)
        self.lens = torch.tensor(case.seq_lens, dtype=torch.int32)

    def oracle(self, batch_index=None, num_splits=None, **mods):
        return int4_cache.decode_int4(
            workloads.to_numpy_f32(self.q), self.kc, self.vc, self.ks, self.vs, self.bt.numpy(),
            np.asarray(self.case.seq_lens), None if self.signs is None else self.signs.numpy(),
            self.scale, num_splits=num_splits, batch_index=batch_index, **mods)

    def to_gpu(self, dev="cuda"):
        g = {}
        g["q"] = self.q.to(dev)
        g["kc"] = torch.from_numpy(self.kc).to(dev)
        g["vc"] = torch.from_numpy(self.vc).to(dev)
        g["ks"] = torch.from_numpy(self.ks.view(np.int32)).to(dev).view(torch.float32)
        g["vs"] = torch.from_numpy(self.vs.view(np.int32)).to(dev).view(torch.float32)
        g["bt"] = self.bt.to(dev)
        g["lens"] = self.lens.to(dev)
        g["signs"] = None if self.signs is None else self.signs.to(dev)
        return g


def assert_close_scaled(gpu, ref, unit, what=""):
    """The attention tolerance on data of magnitude `unit`: (gpu / unit) against (ref / unit)."""
    return assert_close(np.asarray(gpu, np.float64) / unit, np.asarray(ref, np.float64) / unit, what=what)


def run_int4(kvq, g, scale, num_splits=0, out_dtype=torch.float32, **mods):
    out = kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"],
                              scale, num_splits=num_splits, out_dtype=out_dtype, **mods)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0, (st, flags)
    return out


class TqCase:
    def __init__(self, case, value_bits, num_blocks=None):
        self.case = case
        self.bits = value_bits
        self.bt, self.nb = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=num_blocks)
        self.cache = workloads.random_turboquant_slots((self.nb, 16, case.Hk), case.D, value_bits, case.seed)
        self.q = workloads.query(case, dtype=torch.float32)
        self.lens = torch.tensor(case.seq_lens, dtype=torch.int32)
        self.scale = 1.0 / math.sqrt(case.D)

    def oracle(self, batch_index=None):
        return turboquant.decode_tq(self.q.numpy(), self.cache.numpy(), self.bits, self.bt.numpy(),
                                    np.asarray(self.case.seq_lens), self.scale, batch_index=batch_index)


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
        from quantized_paged_kv_int4_gb300 import kvq
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


def scatter_into_pool(cache, bt, num_blocks, seed):
    """cache [n, 16, Hk, sb] (compact pages) placed at random blocks of a num_blocks pool on the GPU,
    the pool's first and last blocks among them; returns (pool, block table into the pool)."""
    n = cache.shape[0]
    g = torch.Generator().manual_seed(seed)
    mid = torch.randperm(num_blocks - 2, generator=g)[:max(n - 2, 0)] + 1
    phys = torch.cat([torch.tensor([num_blocks - 1, 0]), mid])[:n]
    pool = torch.empty((num_blocks,) + tuple(cache.shape[1:]), dtype=torch.uint8, device="cuda")
    pool[phys.cuda()] = cache.cuda()
    return pool, phys[bt.long()].to(torch.int32)
