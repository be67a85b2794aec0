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


@pytest.mark.parametrize("pool", [1, 2, 4, 7, 16])  # 2 and 4: the unrolled kernels
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


def _code_order(c):
    """E4M3FN codes as signed integers ordered like their values (adjacent values differ by 1)."""
    c = np.asarray(c, np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def test_codes_are_within_one_step_of_a_correctly_rounded_exp():
    """The bit-exact checks above use the oracle's written-out fp32 exponential, the same operation
    sequence as the kernel's (the page does not show tl.exp). Against an independent fp32 exp --
    the float64 exponential rounded once (oracle/kpool.py, exp_f32_rounded) -- the kernel's codes
    may differ only where a pooled value sits on a bf16 rounding boundary: each such code by one
    E4M3 step, in at most 1e-4 of all codes, with the same power-of-two scale on every row."""
    n, pool, ps = 16384, 4, 64
    slot_k, score, ape, loc, nb = workloads.kpool_case(n, pool, ps, seed=0)
    g = torch.zeros((nb, ps, 132), dtype=torch.uint8, device="cuda")
    kvq.kvq_kpool_write(g, slot_k.cuda(), score.cuda(), ape.cuda(), loc.cuda())
    assert kvq.kvq_device_error() == (0, 0)
    got = g.cpu().numpy().reshape(nb, ps * 132)
    x = kpool.pool_keys(slot_k.float().numpy(), score.numpy(), ape.numpy(), exp=kpool.exp_f32_rounded)
    codes, scales = kpool.quantize_rows(x)
    page, row = np.divmod(loc.numpy(), ps)
    gpu_codes = np.stack([got[p, r * 128:(r + 1) * 128] for p, r in zip(page, row)])
    gpu_scales = np.array([got[p, ps * 128 + 4 * r:ps * 128 + 4 * r + 4].view(np.float32)[0]
                           for p, r in zip(page, row)])
    assert np.array_equal(gpu_scales, scales)
    step = np.abs(_code_order(gpu_codes) - _code_order(codes))
    assert step.max() <= 1
    assert (step > 0).mean() <= 1e-4, (step > 0).sum()


# ---- tail ring ----------------------------------------------------------------------------------

def _bf16_np(t):
    return t.float().cpu().numpy()


def _tail_views(blocks, ring, pad_blocks=0):
    """A bf16 tail [blocks, 2, ring, 128] inside a larger buffer (padded block stride), NaN-filled."""
    big = torch.full((blocks, 2 * ring * 128 + pad_blocks * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    tail = big[:, :2 * ring * 128].view(blocks, 2, ring, 128)
    return big, tail


def test_seed_tail_bit_exact():
    rng = np.random.default_rng(21)
    ring, kp = 8, 4
    lens = [6, 3, 9, 1, 12]
    tsl = []
    for r, n in enumerate(lens):
        tsl += [r * ring + p % ring for p in range(n)]
    tsl += [-1, -1, -1]
    n = len(tsl)
    key = torch.from_numpy(rng.standard_normal((n, 128)).astype(np.float32)).to(torch.bfloat16)
    score = torch.from_numpy(rng.standard_normal((n, 128)).astype(np.float32)).to(torch.bfloat16)
    big, tail = _tail_views(len(lens), ring, pad_blocks=3)
    ref = _bf16_np(tail)
    kpool.seed_tail(ref, key.float().numpy(), score.float().numpy(), np.array(tsl), kp)
    kvq.kvq_kpool_seed_tail(tail, key.cuda(), score.cuda(), torch.tensor(tsl, dtype=torch.int32, device="cuda"), kp)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0
    got = _bf16_np(tail)
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.array_equal(np.nan_to_num(got), np.nan_to_num(ref))


@pytest.mark.parametrize("next_n,round_scale", [(1, True), (3, True), (4, False)])
def test_decode_update_stream_bit_exact(next_n, round_scale):
    """Prompts seeded into the ring, then decode steps of next_n tokens per request: every cache
    byte and every ring entry equal the oracle's after each step."""
    rng = np.random.default_rng(30 + next_n)
    pool, ring, ps = 4, 8, 16
    prompt, total = [10, 4, 13, 7], [31, 27, 30, 19]
    R = len(prompt)
    keys = [torch.from_numpy(rng.standard_normal((total[r], 128)).astype(np.float32)).to(torch.bfloat16) for r in range(R)]
    scores = [torch.from_numpy(rng.standard_normal((total[r], 128)).astype(np.float32) * 2).to(torch.bfloat16)
              for r in range(R)]
    ape = torch.from_numpy(rng.standard_normal((pool, 128)).astype(np.float32) * 0.5)
    perm = rng.permutation(64 * ps)
    pool_loc, k = {}, 0
    for r in range(R):
        for q in range(total[r] // pool):
            pool_loc[(r, q)] = int(perm[k]); k += 1
    big, tail = _tail_views(R + 1, ring, pad_blocks=1)
    ref_tail = _bf16_np(tail)
    cache = torch.zeros((64, ps, 132), dtype=torch.uint8, device="cuda")
    ref_cache = np.zeros((64, ps, 132), np.uint8)
    tk = torch.cat([keys[r][:prompt[r]] for r in range(R)])
    tsc = torch.cat([scores[r][:prompt[r]] for r in range(R)])
    tsl = [(r + 1) * ring + p % ring for r in range(R) for p in range(prompt[r])]
    kpool.seed_tail(ref_tail, tk.float().numpy(), tsc.float().numpy(), np.array(tsl), pool)
    kvq.kvq_kpool_seed_tail(tail, tk.cuda(), tsc.cuda(), torch.tensor(tsl, dtype=torch.int32, device="cuda"), pool)
    cur = list(prompt)
    while any(cur[r] < total[r] for r in range(R)):
        K = torch.zeros((R, next_n, 128), dtype=torch.bfloat16); S = torch.zeros_like(K)
        P = torch.full((R, next_n), -1, dtype=torch.int32); L = torch.full_like(P, -1); TS = torch.full_like(P, -1)
        for r in range(R):
            for t in range(next_n):
                pos = cur[r] + t
                if pos >= total[r]:
                    continue
                K[r, t], S[r, t], P[r, t] = keys[r][pos], scores[r][pos], pos
                TS[r, t] = (r + 1) * ring + pos % ring
                if pos % pool == pool - 1:
                    L[r, t] = pool_loc[(r, pos // pool)]
        kpool.decode_update(ref_cache, ref_tail, TS.numpy(), K.float().numpy(), S.float().numpy(), ape.numpy(),
                            L.numpy(), P.numpy(), pool, round_scale)
        kvq.kvq_kpool_decode_update(cache, tail, TS.cuda(), K.cuda(), S.cuda(), ape.cuda(), L.cuda(), P.cuda(), pool,
                                    round_scale=round_scale)
        st, flags = kvq.kvq_device_error()
        assert st == 0 and flags == 0
        assert np.array_equal(cache.cpu().numpy(), ref_cache)
        got = _bf16_np(tail)
        assert np.array_equal(np.isnan(got), np.isnan(ref_tail))
        assert np.array_equal(np.nan_to_num(got), np.nan_to_num(ref_tail))
        cur = [min(c + next_n, total[r]) for r, c in enumerate(cur)]
