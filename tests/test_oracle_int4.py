"""Pins for the INT4 write path of the oracle (oracle/int4_cache.py).

Closed-form cases worked by hand from int4_per_token_head.py, _reshape_cache_int4_kernel
(scale = max((max - min) / 15, 1e-6); zp = clamp(round-half-away(-min / scale), 0, 15);
q = clamp(round-half-away(x / scale + zp), 0, 15); word = bits(scale) & ~0xF | zp),
the quantizer's error bound, exhaustive nibble packing and the scatter/gather round trip.
"""

import numpy as np
import torch

from oracle import formats, hadamard, int4_cache
from quantized_paged_kv_int4_gb300 import workloads


def _bits(f):
    return int(np.float32(f).view(np.uint32))


def test_worked_example_symmetric_range():
    # min -7.5, max 7.5 -> scale = 15/15 = 1 exactly; -min/scale = 7.5 -> 7.5 + 0.5 = 8 -> zp 8.
    # x + 8 = [0.5, 6, 8, 15.5] -> round half away from zero -> [1, 6, 8, 16 -> clamp 15].
    # (round-half-even would give 0 for 0.5: this case fixes the rounding rule.)
    q, w = int4_cache.quantize_int4(np.array([[-7.5, -2.0, 0.0, 7.5]], dtype=np.float32))
    assert q.tolist() == [[1, 6, 8, 15]]
    assert int(w[0]) == (_bits(1.0) & ~0xF) | 8 == 0x3F800008


def test_worked_example_one_signed():
    # [2, 3, 4, 5]: scale = fp32(3/15) = fp32(0.2); -2/0.2 = -10 (fp32 -9.99999985 -> -10.4999.. -> -10)
    # -> clamp to zp = 0; 1/fp32(0.2) rounds to 5.0 in fp32; x * 5 = [10, 15, 20, 25] -> clamp -> [10, 15, 15, 15]
    q, w = int4_cache.quantize_int4(np.array([[2.0, 3.0, 4.0, 5.0]], dtype=np.float32))
    assert q.tolist() == [[10, 15, 15, 15]]
    assert np.float32(1.0) / np.float32(3.0 / 15.0) == np.float32(5.0)
    assert int(w[0]) == (_bits(np.float32(3.0) / np.float32(15.0)) & ~0xF)


def test_worked_example_constant_vectors_and_saturation():
    s = np.float32(1e-6)
    # constant 3: scale = 1e-6; -3/1e-6 < 0 -> zp 0; 3 * (1/1e-6) ~ 3e6 -> 15
    q, w = int4_cache.quantize_int4(np.full((1, 8), 3.0, dtype=np.float32))
    assert q.tolist() == [[15] * 8] and int(w[0]) == (_bits(s) & ~0xF)
    # constant -3: -(-3)/1e-6 = 3e6 -> zp = clamp(3e6) = 15; -3e6 + 15 -> 0
    q, w = int4_cache.quantize_int4(np.full((1, 8), -3.0, dtype=np.float32))
    assert q.tolist() == [[0] * 8] and int(w[0]) == (_bits(s) & ~0xF) | 15
    # constant 3000: 3000 * 1e6 = 3e9 exceeds int32; the float->int conversion saturates -> 15
    q, _ = int4_cache.quantize_int4(np.full((1, 8), 3000.0, dtype=np.float32))
    assert q.tolist() == [[15] * 8]
    assert int4_cache.cvt_rzi_sat(np.float32(3e9)) == 2**31 - 1
    assert int4_cache.cvt_rzi_sat(np.float32(-3e9)) == -(2**31)
    assert int4_cache.cvt_rzi_sat(np.float32(np.nan)) == 0
    assert int4_cache.cvt_rzi_sat(np.float32(-2.7)) == -2
    # half-way in fp32: 0.49999997 + 0.5 rounds to 1.0 in fp32, so it rounds up (kept as the pages do it)
    assert int4_cache.round_half_away(np.float32(0.49999997)) == 1
    assert int4_cache.round_half_away(np.float32(-2.5)) == -3


def test_row_of_tens_one_signed_special_case():
    q, _ = int4_cache.quantize_int4(np.full((1, 128), 10.0, dtype=np.float32) + np.float32(0.0))
    assert np.all(q == 15)


def test_pack_unpack_exhaustive():
    b = np.arange(256, dtype=np.uint8)
    nib = int4_cache.unpack_nibbles(b[:, None])
    assert np.array_equal(nib[:, 0], b & 0xF) and np.array_equal(nib[:, 1], b >> 4)
    assert np.array_equal(int4_cache.pack_nibbles(nib)[:, 0], b)
    assert int4_cache.pack_nibbles(np.array([[3, 12]], dtype=np.uint8))[0, 0] == 0xC3


def test_quantizer_invariants_and_error_bound():
    rng = np.random.default_rng(11)
    D = 128
    signs = workloads.rht_signs(D).numpy()
    x = formats.bf16_round(rng.standard_normal((4000, D)).astype(np.float32) * np.float32(rng.uniform(0.01, 50)))
    x[:10, 3] *= np.float32(100.0)  # outliers
    r = int4_cache.rotate_to_bf16(x, signs)
    q, w = int4_cache.quantize_int4(r)
    assert q.max() <= 15
    s, zp = int4_cache.split_scale_word(w)
    assert zp.min() >= 0 and zp.max() <= 15
    assert np.all(s >= np.float64((np.float32(1e-6).view(np.uint32) & ~np.uint32(0xF)).view(np.float32)))
    # the stored scale differs from the true one only in its low 4 mantissa bits
    exact_scale = np.maximum((r.max(1).astype(np.float64) - r.min(1)) / 15.0, 1e-6)
    assert np.all(np.abs(s - exact_scale) <= exact_scale * 2.0**-19)
    deq = int4_cache.dequant_int4(int4_cache.pack_nibbles(q), w)
    mixed = (r.min(1) <= 0) & (r.max(1) >= 0)
    assert mixed.mean() > 0.99
    err = np.abs(deq - r.astype(np.float64))[mixed]
    assert np.all(err <= (s[mixed, None] * (0.5 + 1e-4)))


def test_rotation_matches_matrix_form():
    rng = np.random.default_rng(12)
    D = 128
    signs = workloads.rht_signs(D).numpy().astype(np.float64)
    x = formats.bf16_round(rng.standard_normal((2000, D)).astype(np.float32))
    got = int4_cache.rotate_to_bf16(x, signs.astype(np.float32)).astype(np.float64)
    exact = (x.astype(np.float64) * signs) @ hadamard.sylvester(D).T
    # bf16 of an fp32 sum: equal to bf16(exact) except on a near-tie, where it is one bf16 ulp off
    rnd = formats.bf16_round(exact.astype(np.float32)).astype(np.float64)
    same = got == rnd
    assert same.mean() > 0.999
    ulp = np.abs(rnd) * 2.0**-7
    assert np.all(np.abs(got - rnd)[~same] <= ulp[~same] * 1.01)


def test_write_scatter_gather_round_trip():
    case = workloads.tiny_int4()
    D, Hk = case.D, case.Hk
    bt, nb = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=14, unused_fill=-1)
    seq, pos, slots = workloads.all_token_slots(bt, case.seq_lens)
    T = slots.numel()
    k, v = workloads.kv_vectors(case, T)
    hole = torch.zeros(T, dtype=torch.bool)
    hole[::7] = True
    slots_w = torch.where(hole, torch.full_like(slots, -1), slots)
    kc = np.full((nb, 16, Hk, D // 2), 0xA5, np.uint8)
    vc = np.full((nb, 16, Hk, D // 2), 0x5A, np.uint8)
    ks = np.full((nb, 16, Hk), 0xDEADBEEF, np.uint32)
    vs = np.full((nb, 16, Hk), 0xFEEDFACE, np.uint32)
    signs = workloads.rht_signs(D).numpy()
    kf, vf = workloads.to_numpy_f32(k), workloads.to_numpy_f32(v)
    int4_cache.write_int4(kf, vf, slots_w.numpy(), signs, kc, vc, ks, vs)
    # untouched slots keep their sentinel bytes
    written = np.zeros((nb * 16,), bool)
    written[slots_w[slots_w >= 0].numpy()] = True
    wmask = written.reshape(nb, 16)
    assert np.all(kc[~wmask] == 0xA5) and np.all(vs[~wmask] == 0xFEEDFACE)
    # every written token, gathered back through the block table position by position
    for t in range(T):
        if hole[t]:
            continue
        b, n = int(seq[t]), int(pos[t])
        page, row = int(bt[b, n // 16]), n % 16
        for src, cache, sc in ((kf, kc, ks), (vf, vc, vs)):
            r = int4_cache.rotate_to_bf16(src[t], signs)
            deq = int4_cache.dequant_int4(cache[page, row], sc[page, row])
            s, _ = int4_cache.split_scale_word(sc[page, row])
            assert np.all(np.abs(deq - r) <= s[:, None] * (0.5 + 1e-4))
