"""Pins for the oracle's kpool compress-and-write (oracle/kpool.py; kpool_compress.py,
_kpool_softmax_rotate_write_cache_kernel): its fp32 exponential against math.exp, pools that
reduce to one key or to an exact mean (then the result is the pinned FWHT-128 FP8 quantizer's),
the unrounded scale mapping the absmax to +-448, and the paged scatter."""

import math

import numpy as np
import pytest

from oracle import fwht_fp8, kpool, formats
from quantized_paged_kv_int4_gb300 import workloads

F32 = np.float32


def _ulp_diff(a, b):
    ia = np.asarray(a, F32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, F32).view(np.int32).astype(np.int64)
    return np.abs(ia - ib)


def test_exp_f32_against_math_exp():
    rng = np.random.default_rng(1)
    x = np.concatenate([-rng.random(20000).astype(F32) * 80, -rng.random(20000).astype(F32),
                        np.array([0.0, -1e-8, -0.5, -1.0, -87.0, -88.7, -103.0], F32)]).astype(F32)
    ref = np.array([F32(math.exp(float(v))) for v in x], F32)
    normal = ref >= F32(2.0 ** -125)
    assert _ulp_diff(kpool.exp_f32(x)[normal], ref[normal]).max() <= 1
    assert np.all(kpool.exp_f32(x)[ref < F32(2.0 ** -127)] == 0.0)   # flushed below the normal range
    assert kpool.exp_f32(np.array([0.0], F32))[0] == 1.0
    assert kpool.exp_f32(np.array([-np.inf, -1e30], F32)).tolist() == [0.0, 0.0]


def _bf16(rng, shape, scale=1.0):
    return formats.bf16_round((rng.standard_normal(shape) * scale).astype(F32))


def test_pool_of_one_is_the_fwht_fp8_quantizer():
    rng = np.random.default_rng(2)
    k = _bf16(rng, (6, 1, 128))
    score = rng.standard_normal((6, 1, 128)).astype(F32)
    ape = rng.standard_normal((1, 128)).astype(F32)
    codes, scales = kpool.quantize_rows(kpool.pool_keys(k, score, ape))
    ref_codes, ref_scales = fwht_fp8.fwht128_quant_fp8(k[:, 0])
    assert np.array_equal(codes, ref_codes) and np.array_equal(scales, ref_scales)


def test_equal_scores_give_the_exact_mean():
    """Equal scores -> weights 1 each; keys on a coarse grid make the fp32 sum and the division by
    the pool size exact, so x is the mean exactly."""
    rng = np.random.default_rng(3)
    k = (rng.integers(-64, 64, size=(5, 4, 128)) / 16.0).astype(F32)
    score = np.full((5, 4, 128), 0.25, F32)
    ape = np.zeros((4, 128), F32)
    x = kpool.pool_keys(k, score, ape)
    assert np.array_equal(x, formats.bf16_round(k.mean(axis=1).astype(F32)))
    codes, scales = kpool.quantize_rows(x)
    ref = fwht_fp8.fwht128_quant_fp8(x)
    assert np.array_equal(codes, ref[0]) and np.array_equal(scales, ref[1])


def test_dominant_slot_selects_its_key():
    rng = np.random.default_rng(4)
    k = _bf16(rng, (3, 8, 128), 2.0)
    score = rng.standard_normal((3, 8, 128)).astype(F32)
    score[:, 5] += 200.0  # e^-190 underflows: every other weight is 0
    x = kpool.pool_keys(k, score, np.zeros((8, 128), F32))
    assert np.array_equal(x, k[:, 5])


def test_unrounded_scale_maps_the_absmax_to_448():
    rng = np.random.default_rng(5)
    x = _bf16(rng, (16, 128))
    codes, scales = kpool.quantize_rows(x, round_scale=False)
    y = formats.bf16_round(kpool.hadamard128_normalised_f32(x))
    a = np.maximum(np.abs(y).max(axis=1), F32(1e-4))
    assert np.array_equal(scales, (a * F32(1.0 / 448.0)).astype(F32))
    i = np.abs(y).argmax(axis=1)
    assert np.all(np.isin(codes[np.arange(16), i], [0x7E, 0xFE]))   # +-448


def test_scatter_to_pages_and_write_mask():
    rng = np.random.default_rng(6)
    n, P, ps = 7, 4, 16
    cache = np.full((5, ps, 132), 0xA5, np.uint8)
    k = _bf16(rng, (n, P, 128))
    score = rng.standard_normal((n, P, 128)).astype(F32)
    ape = rng.standard_normal((P, 128)).astype(F32)
    loc = np.array([3, 17, 79, 40, 0, 63, 31], np.int64)
    mask = np.array([1, 1, 0, 1, 1, 1, 0], bool)
    codes, scales = kpool.kpool_compress_write(cache, k, score, ape, loc, mask)
    flat = cache.reshape(5, ps * 132)
    for p in range(n):
        page, off = divmod(int(loc[p]), ps)
        got_k = flat[page, off * 128:(off + 1) * 128]
        got_s = flat[page, ps * 128 + 4 * off:ps * 128 + 4 * off + 4]
        if mask[p]:
            assert np.array_equal(got_k, codes[p])
            assert got_s.tobytes() == scales[p].tobytes()
        else:
            assert np.all(got_k == 0xA5) and np.all(got_s == 0xA5)
    assert (flat != 0xA5).sum() == 5 * (128 + 4)   # nothing else touched


# ---- tail ring (prefill seeding + batched decode update) --------------------------------------

def _stream(R=3, pool=4, ring=8, next_n=3, seed=7):
    """R requests with prompts of different lengths, then decode steps of next_n tokens each."""
    rng = np.random.default_rng(seed)
    prompt = [10, 4, 13][:R]
    total = [31, 27, 30][:R]
    keys = [_bf16(rng, (total[r], 128)) for r in range(R)]
    scores = [formats.bf16_round(rng.standard_normal((total[r], 128)).astype(F32) * 2) for r in range(R)]
    ape = rng.standard_normal((pool, 128)).astype(F32) * 0.5
    n_slots = 64 * 16
    perm = rng.permutation(n_slots)
    pool_loc = {}
    for r in range(R):
        for q in range(total[r] // pool):
            pool_loc[(r, q)] = int(perm[len(pool_loc)])
    return prompt, total, keys, scores, ape, pool_loc, pool, ring, next_n


def test_decode_update_reproduces_direct_pool_compression():
    """Seeding the prompts' tails, then feeding the rest next_n tokens at a time through the ring,
    writes every pool completed during decode exactly as compressing that pool directly."""
    prompt, total, keys, scores, ape, pool_loc, pool, ring, next_n = _stream()
    R = len(prompt)
    tail = np.full((R + 2, 2, ring, 128), np.nan, F32)   # tail block r + 1 (block 0 unused)
    # prefill: all prompt tokens of the batch, flattened
    tk, ts, tsl = [], [], []
    for r in range(R):
        for pos in range(prompt[r]):
            tk.append(keys[r][pos]); ts.append(scores[r][pos]); tsl.append((r + 1) * ring + pos % ring)
    tsl.append(-1)  # padding
    tk.append(np.zeros(128, F32)); ts.append(np.zeros(128, F32))
    kpool.seed_tail(tail, np.array(tk), np.array(ts), np.array(tsl), pool)
    cache = np.zeros((64, 16, 132), np.uint8)
    cur = list(prompt)
    while any(cur[r] < total[r] for r in range(R)):
        K = np.zeros((R, next_n, 128), F32); S = np.zeros_like(K)
        P = np.full((R, next_n), -1, np.int64); L = np.full((R, next_n), -1, np.int64)
        TS = np.full((R, next_n), -1, np.int64)
        for r in range(R):
            for t in range(next_n):
                pos = cur[r] + t
                if pos >= total[r]:
                    continue
                K[r, t], S[r, t], P[r, t] = keys[r][pos], scores[r][pos], pos
                TS[r, t] = (r + 1) * ring + pos % ring
                if pos % pool == pool - 1:
                    L[r, t] = pool_loc[(r, pos // pool)]
        kpool.decode_update(cache, tail, TS, K, S, ape, L, P, pool)
        cur = [min(c + next_n, total[r]) for r, c in enumerate(cur)]
    flat = cache.reshape(64, 16 * 132)
    checked = 0
    for (r, q), loc in pool_loc.items():
        if (q + 1) * pool - 1 < prompt[r]:
            continue  # completed in the prompt: written by the prefill compress, not here
        codes, scales = kpool.quantize_rows(kpool.pool_keys(keys[r][None, q * pool:(q + 1) * pool],
                                                            scores[r][None, q * pool:(q + 1) * pool], ape))
        page, off = divmod(loc, 16)
        assert np.array_equal(flat[page, off * 128:(off + 1) * 128], codes[0])
        assert flat[page, 16 * 128 + 4 * off:16 * 128 + 4 * off + 4].tobytes() == scales[0].tobytes()
        checked += 1
    assert checked >= 12


def test_seed_tail_copies_only_each_requests_last_kpool_tokens():
    rng = np.random.default_rng(8)
    ring, kpool_n = 8, 4
    lens = [6, 3, 9]
    tsl, owner = [], []
    for r, n in enumerate(lens):
        for pos in range(n):
            tsl.append(r * ring + pos % ring); owner.append((r, pos))
    tsl += [-1, -1]
    owner += [None, None]
    key = rng.standard_normal((len(tsl), 128)).astype(F32)
    score = rng.standard_normal((len(tsl), 128)).astype(F32)
    tail = np.full((3, 2, ring, 128), 7.0, F32)
    kpool.seed_tail(tail, key, score, np.array(tsl), kpool_n)
    expect = np.full_like(tail, 7.0)
    for i, o in enumerate(owner):
        if o is not None and o[1] >= lens[o[0]] - kpool_n:
            expect[o[0], 0, o[1] % ring] = key[i]
            expect[o[0], 1, o[1] % ring] = score[i]
    assert np.array_equal(tail, expect)


def test_written_out_exp_and_a_correctly_rounded_exp_pool_alike():
    """The choice of fp32 exponential (the page does not show tl.exp's) moves a pooled bf16 value
    only when it sits on a rounding boundary: against exp rounded once from float64, at most one
    bf16 ulp, in a handful of 2.1 million values."""
    slot_k, score, ape, loc, nb = workloads.kpool_case(4096, 4, 64, seed=3)
    k = workloads.to_numpy_f32(slot_k)
    x1 = kpool.pool_keys(k, score.numpy(), ape.numpy())
    x2 = kpool.pool_keys(k, score.numpy(), ape.numpy(), exp=kpool.exp_f32_rounded)
    u1 = (x1.view(np.uint32) >> 16).astype(np.int64)
    u2 = (x2.view(np.uint32) >> 16).astype(np.int64)
    assert np.all(np.sign(x1) == np.sign(x2))
    assert np.abs(u1 - u2).max() <= 1
    assert (u1 != u2).mean() <= 1e-4
    assert np.max(np.abs(kpool.exp_f32_rounded(np.float32(-1.0)) - np.float32(np.exp(-1.0)))) == 0
