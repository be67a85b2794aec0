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


# ---- MSE keys (_tq_decode_stage1 with KEY_FP8 = 0) ----------------------------------------------

def _mse_case(key_bits, value_bits, D=64, Hk=2, G=2, lens=(13, 40), seed=31):
    mse, kps, sb = workloads.turboquant_mse_layout(D, key_bits, value_bits)
    bt, nb = workloads.paged_layout(list(lens), seed)
    cache = workloads.random_turboquant_mse_slots((nb, 16, Hk), D, key_bits, value_bits, seed).numpy()
    q = workloads.query(workloads.DecodeCase("m", len(lens), Hk * G, Hk, D, list(lens), seed=seed),
                        dtype=torch.float32).numpy()
    cb = workloads.mse_codebook(key_bits, D).numpy()
    return dict(cache=cache, q=q, cb=cb, bt=bt.numpy(), lens=np.array(lens), mse=mse, kps=kps, D=D, Hk=Hk, G=G)


def _keys_by_unpackbits(cache, key_bits, D, cb, mse, corr):
    """Keys from np.unpackbits (little bit order): an independent unpacking of the index stream."""
    bits = np.unpackbits(cache[..., :mse], axis=-1, bitorder="little")[..., :D * key_bits]
    bits = bits.reshape(bits.shape[:-1] + (D, key_bits)).astype(np.int64)
    idx = (bits << np.arange(key_bits)).sum(axis=-1)
    c = cb.astype(np.float64)[idx]
    if corr:
        c = c / np.sqrt((c * c).sum(axis=-1, keepdims=True) + 1e-16)
    norm = formats.fp16_to_f64(cache[..., mse].astype(np.uint16) | (cache[..., mse + 1].astype(np.uint16) << 8))
    return c * norm[..., None]


def test_mse_bit_stream_worked_example():
    # indices 0..7 at 3 bits each, LSB first: the stream is the integer sum idx_d << 3d
    stream = sum(d << (3 * d) for d in range(8)).to_bytes(3, "little")
    slot = np.frombuffer(stream + b"\x00\x00", dtype=np.uint8)[None]
    assert turboquant._bit_field(slot, 0, 8, 3)[0].tolist() == list(range(8))
    slot = np.frombuffer(bytes([0x10, 0x32, 0x54, 0x76, 0]), dtype=np.uint8)[None]
    assert turboquant._bit_field(slot, 0, 8, 4)[0].tolist() == list(range(8))


@pytest.mark.parametrize("key_bits,value_bits,corr", [(3, 4, False), (4, 3, True), (3, 3, True), (4, 4, False)])
def test_mse_decode_matches_sdpa_with_the_rotation_on_the_keys(key_bits, value_bits, corr):
    """q_rot . c = (q Pi^T) . c = q . (c Pi): SDPA on the original query with keys rotated back."""
    c = _mse_case(key_bits, value_bits)
    D, Hk, G = c["D"], c["Hk"], c["G"]
    Pi = workloads.random_rotation(D, 7).numpy()
    scale = 0.7
    got = turboquant.decode_tq_mse(c["q"], c["cache"], key_bits, c["kps"], value_bits, c["cb"], corr, Pi,
                                   c["bt"], c["lens"], scale)
    for b, L in enumerate(c["lens"]):
        n = np.arange(L)
        slots = c["cache"][c["bt"][b][n // 16], n % 16]                       # [L, Hk, slot]
        K = _keys_by_unpackbits(slots, key_bits, D, c["cb"], c["mse"], corr) @ Pi.astype(np.float64)
        V = turboquant.dequant_values(slots, D, value_bits, c["kps"])
        Q = torch.from_numpy(c["q"][b].astype(np.float64))[:, None, :]           # [Hq, 1, D]
        Kt = torch.from_numpy(np.repeat(K.transpose(1, 0, 2), G, axis=0))
        Vt = torch.from_numpy(np.repeat(V.transpose(1, 0, 2), G, axis=0))
        exp = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, scale=scale)[:, 0].numpy()
        assert np.max(np.abs(got[b] - exp)) < 1e-10


def test_mse_norm_correction_and_codebook_scale():
    """Scaling the codebook by a = 4: with NORM_CORRECTION nothing changes; without it the scores
    scale by a (compensated by attn_scale / a)."""
    c = _mse_case(4, 4, seed=32)
    Pi = workloads.random_rotation(c["D"], 8).numpy()
    run = lambda cb, corr, sc: turboquant.decode_tq_mse(c["q"], c["cache"], 4, c["kps"], 4, cb, corr, Pi,
                                                      c["bt"], c["lens"], sc)
    a = np.float32(4.0)  # a power of two: the scaled codebook is exact in fp32
    assert np.max(np.abs(run(c["cb"] * a, True, 0.5) - run(c["cb"], True, 0.5))) < 1e-12
    assert np.max(np.abs(run(c["cb"] * a, False, 0.5 / 4.0) - run(c["cb"], False, 0.5))) < 1e-12
    assert np.max(np.abs(run(c["cb"], True, 0.5) - run(c["cb"], False, 0.5))) > 1e-6


def test_mse_identity_rotation_zero_query_is_uniform_mean():
    c = _mse_case(3, 4, seed=33)
    q = np.zeros_like(c["q"])
    got = turboquant.decode_tq_mse(q, c["cache"], 3, c["kps"], 4, c["cb"], False, np.eye(c["D"], dtype=np.float32),
                                   c["bt"], c["lens"], 1.0)
    for b, L in enumerate(c["lens"]):
        n = np.arange(L)
        V = turboquant.dequant_values(c["cache"][c["bt"][b][n // 16], n % 16], c["D"], 4, c["kps"])
        assert np.max(np.abs(got[b] - np.repeat(V.mean(axis=0), c["G"], axis=0))) < 1e-12


def test_tq_lse_of_a_zero_query_is_the_log_of_the_length():
    """Every score is 0: lse = ln L exactly; an empty row is -inf."""
    case = workloads.DecodeCase("tql", 3, 4, 2, 64, [20, 0, 7], seed=25)
    bt, nb = workloads.paged_layout(case.seq_lens, case.seed)
    cache = workloads.random_turboquant_slots((nb, 16, 2), 64, 4, case.seed).numpy()
    q = np.zeros((3, 4, 64), np.float32)
    _, lse = turboquant.decode_tq(q, cache, 4, bt.numpy(), np.array(case.seq_lens), 0.125, return_lse=True)
    assert np.allclose(lse[0], np.log(20.0), atol=1e-12) and np.allclose(lse[2], np.log(7.0), atol=1e-12)
    assert np.all(lse[1] == -np.inf)
