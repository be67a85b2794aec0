"""Pins for oracle/turboquant.py: bit-level unpacking against an independent bit writer,
dequantization against the generating values, and attention against torch's SDPA."""

import numpy as np
import pytest
import torch

from oracle import formats, turboquant
from quantized_paged_kv_int4_gb300 import workloads


def _bitwise_pack3(idx, D):
    """Write 3-bit indices one bit at a time into an LSB-first stream (independent writer)."""
    out = np.zeros(idx.shape[:-1] + (-(-3 * D // 8),), np.uint8)
    for d in range(D):
        for j in range(3):
            bit = 3 * d + j
            out[..., bit // 8] |= (((idx[..., d] >> j) & 1) << (bit % 8)).astype(np.uint8)
    return out


@pytest.mark.parametrize("bits", [3, 4])
def test_value_index_unpacking(bits):
    rng = np.random.default_rng(bits)
    D = 128
    idx = rng.integers(0, 1 << bits, size=(50, D))
    slot = workloads.turboquant_slot_bytes(D, bits)
    s = np.zeros((50, slot), np.uint8)
    vdb = -(-D * bits // 8)
    if bits == 4:
        s[:, D:D + vdb] = (idx[:, 0::2] | (idx[:, 1::2] << 4)).astype(np.uint8)
    else:
        s[:, D:D + vdb] = _bitwise_pack3(idx, D)
    # scale 1.0 (0x3C00), zero 0.0 -> values are the indices
    s[:, D + vdb] = 0x00
    s[:, D + vdb + 1] = 0x3C
    _, v = turboquant.dequant_slots(s, D, bits)
    assert np.array_equal(v, idx.astype(np.float64))
    assert slot == (208 if bits == 4 else 192)


@pytest.mark.parametrize("bits", [3, 4])
def test_dequant_matches_generated_values(bits):
    D = 128
    k = torch.randn((40, D)) * 3
    v = torch.randn((40, D))
    slots = workloads.random_turboquant_slots((40,), D, bits, seed=1, k=k, v=v).numpy()
    kd, vd = turboquant.dequant_slots(slots, D, bits)
    assert np.array_equal(kd, k.to(torch.float8_e4m3fn).to(torch.float64).numpy())
    vdb = -(-D * bits // 8)
    sc = formats.fp16_to_f64(slots[:, D + vdb].astype(np.uint16) | (slots[:, D + vdb + 1].astype(np.uint16) << 8))
    # reconstruction within half a grid step (plus fp16 rounding of zero / scale)
    err = np.abs(vd - v.numpy().astype(np.float64))
    assert np.all(err <= sc[:, None] * 0.5 + 2e-3)


@pytest.mark.parametrize("bits", [3, 4])
def test_decode_matches_sdpa(bits):
    B, Hq, Hk, D = 3, 8, 2, 128
    lens = [1, 35, 64]
    bt, nb = workloads.paged_layout(lens, 2, num_blocks=10, unused_fill=-1)
    cache = workloads.random_turboquant_slots((nb, 16, Hk), D, bits, seed=2).numpy()
    q = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(3))
    scale = 1.0 / np.sqrt(D)
    got = turboquant.decode_tq(q.numpy(), cache, bits, bt.numpy(), np.array(lens), scale)
    for b, L in enumerate(lens):
        K = np.zeros((L, Hk, D))
        V = np.zeros((L, Hk, D))
        for n in range(L):
            K[n], V[n] = turboquant.dequant_slots(cache[bt[b, n // 16], n % 16], D, bits)
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(Hq // Hk, 0)[None]
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(Hq // Hk, 0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b].to(torch.float64)[None, :, None, :], Kt, Vt, scale=scale)[0, :, 0, :].numpy()
        assert np.max(np.abs(got[b] - o)) < 1e-12
