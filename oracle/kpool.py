"""kpool compress-and-write: pooled softmax-weighted key -> Hadamard-128 -> FP8 -> paged write.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source page: kpool_compress.py, _kpool_softmax_rotate_write_cache_kernel and
kpool_compress_and_write_cache. Per pool p (one cache entry for pool_size consecutive tokens),
per dimension d, in fp32:
  1. z_s = slot_score[p, s, d] + ape[s, d];  M = max_s z_s
  2. w_s = exp(z_s - M);  den = sum_s w_s;  acc = sum_s slot_k[p, s, d] * w_s  (slot order)
  3. x = bf16(acc / den)  (zero when the pool is masked out)
  4. y = bf16(FWHT_128(x) * fp32(1/sqrt(128)))  (stages h = 1 .. 64, as fwht_fp8)
  5. a = max(max_d |y|, 1e-4); scale = smallest power of two >= a * fp32(1/448) when round_scale,
     else a * fp32(1/448); code = E4M3FN(clamp(y / scale, -448, 448))
  6. cache page loc // page_size: the 128 codes at row loc % page_size, the fp32 scale in the
     page's scale area after page_size * 128 bytes.
Readings: `acc += k * prob` is a multiply then an add (no fused multiply-add); exp is an fp32
exponential -- the page's tl.exp is not shown; here it is exp_f32 below, the same fp32
operation sequence the library uses, so both sides round the pooled value identically before
the quantizer's integer decisions.
"""

import math

import numpy as np

from .formats import bf16_round, f32_to_e4m3fn
from .fwht_fp8 import pow2_ceil
from .hadamard import hadamard128_normalised_f32

F32 = np.float32

# Cody and Waite's range reduction (Software Manual for the Elementary Functions, 1980): x = n ln2 + r
# with ln2 split into LN2_HI (trailing 12 mantissa bits zero, so n * LN2_HI is exact for |n| < 2^11)
# and LN2_LO; e^r for |r| <= ln2 / 2 by the Taylor series to degree 7 (remainder < 1e-8 relative).
_LN2_HI = F32(np.frombuffer((np.float32(0.6931471805599453).view(np.uint32) & np.uint32(0xFFFFF000)).tobytes(),
                            np.float32)[0])
_LN2_LO = F32(0.6931471805599453 - float(_LN2_HI))
_EXP_COEF = [F32(1.0 / math.factorial(k)) for k in range(8)]
_LOG2E = F32(1.4426950408889634)


def exp_f32(x):
    """exp(x) for fp32 x <= 0 in fp32 operations, each rounded to nearest (no fused ops):
    n = rint(x * log2 e); r = (x - n * LN2_HI) - n * LN2_LO; e^r by Horner on the Taylor
    coefficients; times 2^n (ldexp, exact). Results that would fall below the normal range
    (n <= -126, x below about -87) are flushed to 0, as is -inf."""
    x = np.maximum(np.asarray(x, dtype=F32), F32(-104.0))
    n = np.rint((x * _LOG2E).astype(F32)).astype(F32)
    r = ((x - (n * _LN2_HI).astype(F32)).astype(F32) - (n * _LN2_LO).astype(F32)).astype(F32)
    p = np.full_like(r, _EXP_COEF[7])
    for c in _EXP_COEF[6::-1]:
        p = ((p * r).astype(F32) + c).astype(F32)
    out = np.ldexp(p, np.maximum(n, F32(-125.0)).astype(np.int32)).astype(F32)
    return np.where(n <= F32(-126.0), F32(0.0), out).astype(F32)


def exp_f32_rounded(x):
    """exp(x) rounded once to fp32 from the float64 exponential (within half an fp32 ulp but for
    rare double-rounding ties): an fp32 exponential independent of exp_f32's operation sequence,
    the checker for the choice of exp (the page does not show tl.exp's)."""
    with np.errstate(under="ignore"):
        return np.exp(np.asarray(x, dtype=F32).astype(np.float64)).astype(F32)


def pool_keys(slot_k, slot_score, ape, exp=exp_f32):
    """Steps 1-3 without the mask: [n_pools, 128] fp32 holding bf16 values (exp: the fp32
    exponential used for w_s)."""
    k = np.asarray(slot_k, dtype=F32)
    z = (np.asarray(slot_score, dtype=F32) + np.asarray(ape, dtype=F32)[None]).astype(F32)
    M = z.max(axis=1)
    den = np.zeros_like(M)
    acc = np.zeros_like(M)
    for s in range(k.shape[1]):  # slot order, as the page's static loop
        w = exp((z[:, s] - M).astype(F32))
        den = (den + w).astype(F32)
        acc = (acc + (k[:, s] * w).astype(F32)).astype(F32)
    return bf16_round((acc / den).astype(F32))


def quantize_rows(x, round_scale=True):
    """Steps 4-5: (codes uint8 [n, 128], scale float32 [n])."""
    y = bf16_round(hadamard128_normalised_f32(np.asarray(x, dtype=F32)))
    a = np.maximum(np.abs(y).max(axis=1), F32(1e-4)) if y.shape[0] else np.zeros((0,), F32)
    m = (a * F32(1.0 / 448.0)).astype(F32)
    s = pow2_ceil(m) if round_scale else m
    q = np.clip((y / s[:, None]).astype(F32), F32(-448.0), F32(448.0)).astype(F32)
    return f32_to_e4m3fn(q), s.astype(F32)


def kpool_compress_write(kv_cache, slot_k, slot_score, ape, loc, write_mask=None, round_scale=True,
                         exp=exp_f32):
    """kv_cache: uint8 [num_blocks, page_size, 128 + 4] written in place; returns (codes, scales)
    of every pool (masked pools quantize a zero vector and are not written)."""
    n = np.asarray(slot_k).shape[0]
    x = pool_keys(slot_k, slot_score, ape, exp=exp)
    if write_mask is not None:
        x = np.where(np.asarray(write_mask, bool)[:, None], x, F32(0.0)).astype(F32)
    codes, scales = quantize_rows(x, round_scale)
    nb, ps, row = kv_cache.shape
    flat = kv_cache.reshape(nb, ps * row)
    for p in range(n):
        if write_mask is not None and not write_mask[p]:
            continue
        page, off = divmod(int(loc[p]), ps)
        flat[page, off * 128:(off + 1) * 128] = codes[p]
        flat[page, ps * 128 + 4 * off:ps * 128 + 4 * off + 4] = np.frombuffer(scales[p].tobytes(), np.uint8)
    return codes, scales


# ----------------------------------------------------------------------------------------------
# tail ring: prefill seeding and the batched decode-step update
# ----------------------------------------------------------------------------------------------


def seed_tail(tail, key, gate_score, tslot, kpool):
    """kpool_compress.py, _kpool_tail_seed_kernel. tail: [num_blocks, 2, ring, 128] float32 holding
    bf16 values (half 0 keys, half 1 scores), written in place; key / gate_score [n, 128] (bf16
    values); tslot [n] int (block * ring + pos % ring, < 0 = padding). Token i is copied iff it is
    one of its request's last kpool tokens: the token kpool ahead is past the batch, padding, or
    in another tail block."""
    ring = tail.shape[2]
    n = len(tslot)
    for i in range(n):
        t = int(tslot[i])
        if t < 0:
            continue
        blk = t // ring
        ahead = int(tslot[i + kpool]) if i + kpool < n else -1
        if ahead >= 0 and ahead // ring == blk:
            continue
        tail[blk, 0, t % ring] = key[i]
        tail[blk, 1, t % ring] = gate_score[i]


def decode_update(kv_cache, tail, tail_slot, key, slot_score, ape, slot_mapping, positions, pool_size,
                  round_scale=True):
    """kpool_compress.py, _kpool_decode_update_batched_kernel: per request, its next_n tokens in
    order. Token (r, t) with pos = positions[r, t] >= 0:
      * if slot_mapping[r, t] >= 0 and pos % pool_size == pool_size - 1, the pool ending at pos is
        compressed -- its earlier slots from the tail ring (phys = (pos - slot + j) % ring), its
        last one the current key / score -- with the pooled softmax + Hadamard + FP8 of
        kpool_compress_write and written at slot_mapping[r, t];
      * then, if tail_slot[r, t] >= 0, the current key and score are stashed at ring position
        pos % ring of block tail_slot[r, t] // ring.
    tail: [num_blocks, 2, ring, 128] float32 (bf16 values), kv_cache: uint8 [nb, page_size, 132],
    both written in place."""
    ring = tail.shape[2]
    R, T = positions.shape
    nb, ps, _ = kv_cache.shape
    flat = kv_cache.reshape(nb, ps * 132)
    ape = np.asarray(ape, F32)
    for r in range(R):
        for t in range(T):
            pos = int(positions[r, t])
            loc = int(slot_mapping[r, t])
            ts = int(tail_slot[r, t])
            blk = max(ts, 0) // ring
            slot = max(pos, 0) % pool_size
            if loc >= 0 and pos >= 0 and slot == pool_size - 1:
                start = pos - slot
                ks = np.empty((1, pool_size, 128), F32)
                ss = np.empty((1, pool_size, 128), F32)
                for j in range(pool_size):
                    phys = (start + j) % ring
                    cur = j == slot
                    ks[0, j] = key[r, t] if cur else tail[blk, 0, phys]
                    ss[0, j] = slot_score[r, t] if cur else tail[blk, 1, phys]
                codes, scales = quantize_rows(pool_keys(ks, ss, ape), round_scale)
                page, off = divmod(loc, ps)
                flat[page, off * 128:(off + 1) * 128] = codes[0]
                flat[page, ps * 128 + 4 * off:ps * 128 + 4 * off + 4] = np.frombuffer(scales[0].tobytes(), np.uint8)
            if pos >= 0 and ts >= 0:
                tail[blk, 0, pos % ring] = key[r, t]
                tail[blk, 1, pos % ring] = slot_score[r, t]
