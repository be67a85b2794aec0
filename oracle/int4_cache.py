"""INT4 per-(token, head) paged KV cache: write, dequantize, decode attention.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source page: int4_per_token_head.py (tduncan/Nvidia-Optimization-Stack-VLLM).

Write (reshape_and_cache_int4 -> _reshape_cache_int4_kernel), per token t whose
slot_mapping entry is >= 0 and per kv-head h, for K and V independently:
  1. r = bf16(H(x * d1)) -- single_rht of the fp32 vector, cast back to the input
     dtype (bf16), with the fp32 butterfly of fast_hadamard_transform;
  2. mn = min r, mx = max r, scale = max((mx - mn) / 15, 1e-6);
  3. zp = clamp(int(round-half-away(-mn / scale)), 0, 15), where round-half-away(t)
     is trunc(t + 0.5) for t >= 0 and trunc(t - 0.5) otherwise;
  4. q_i = clamp(round-half-away(r_i * (1 / scale) + zp), 0, 15);
  5. byte j = q_{2j} | q_{2j+1} << 4 (pack_int4_nibbles);
  6. scale word = (bits(scale) & ~0xF) | zp, the zero-point hidden in the low four
     mantissa bits of the fp32 scale;
  7. stored at page slot_mapping[t] // block_size, row slot_mapping[t] % block_size.
All of it in IEEE fp32 with one rounding per written operation (no fused
multiply-add), float -> int32 truncating toward zero and saturating (NaN -> 0).

Read (_attn_packed): the scale word gives zp = w & 0xF and scale' = float(w & ~0xF);
a stored nibble q dequantizes to (q - zp) * scale'. unified_attention_int4 rotates
q the same way as the cache (q_rot = bf16(H(q * d1))), divides the softmax scale
by D (the forward RHT has norm sqrt(D)) and maps the output back with
H(o) * d1 / D. Here the attention itself is evaluated in float64 on the
dequantized cache: softmax(sm * q_rot . k) weighted sum of v.
"""

import numpy as np

from .formats import bf16_round
from .hadamard import rht_forward, rht_inverse_f64

F32 = np.float32
INT32_MAX = 2**31 - 1
INT32_MIN = -(2**31)


def cvt_rzi_sat(x):
    """float32 -> int32: truncate toward zero, saturate at the int32 range, NaN -> 0."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    t = np.trunc(np.nan_to_num(x, nan=0.0, posinf=np.inf, neginf=-np.inf))
    t = np.clip(t, INT32_MIN, INT32_MAX)
    return t.astype(np.int64)


def round_half_away(x):
    """The pages' rounding: where(x >= 0, int(x + 0.5), int(x - 0.5)), all in fp32."""
    x = np.asarray(x, dtype=np.float32)
    up = cvt_rzi_sat(x + F32(0.5))
    down = cvt_rzi_sat(x - F32(0.5))
    return np.where(x >= 0, up, down)


def quantize_int4(r):
    """Asymmetric INT4 quantization of bf16-valued fp32 vectors along the last axis.

    Returns (nibbles uint8 [..., D], scale word uint32 [...]).
    """
    r = np.asarray(r, dtype=np.float32)
    mn = r.min(axis=-1)
    mx = r.max(axis=-1)
    scale = np.maximum((mx - mn) / F32(15.0), F32(1e-6)).astype(np.float32)
    t = (-mn) / scale
    zp = np.clip(round_half_away(t).astype(np.float32), F32(0.0), F32(15.0))
    inv = F32(1.0) / scale
    prod = r * inv[..., None]            # rounded to fp32
    u = prod + zp[..., None]             # rounded to fp32 again
    q = np.clip(round_half_away(u).astype(np.float32), F32(0.0), F32(15.0))
    word = (scale.view(np.uint32) & np.uint32(0xFFFFFFF0)) | (
        zp.astype(np.int64).astype(np.uint32) & np.uint32(0xF))
    return q.astype(np.uint8), word.astype(np.uint32)


def pack_nibbles(q):
    """Byte j holds element 2j in its low nibble and element 2j+1 in its high nibble."""
    q = np.asarray(q, dtype=np.uint8)
    return ((q[..., 0::2] & 0xF) | ((q[..., 1::2] & 0xF) << 4)).astype(np.uint8)


def unpack_nibbles(b):
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = (b >> 4) & 0xF
    return out


def split_scale_word(word):
    """(scale' as float64, zp as int64) from the packed fp32 scale word."""
    w = np.asarray(word, dtype=np.uint32)
    zp = (w & np.uint32(0xF)).astype(np.int64)
    scale = (w & np.uint32(0xFFFFFFF0)).view(np.float32).astype(np.float64)
    return scale, zp


def dequant_int4(packed, word):
    """(q - zp) * scale' in float64, packed [..., D/2] uint8, word [...] uint32."""
    q = unpack_nibbles(packed).astype(np.float64)
    scale, zp = split_scale_word(word)
    return (q - zp[..., None]) * scale[..., None]


def rotate_to_bf16(x, signs):
    """bf16(H(x * d1)) of bf16-valued fp32 vectors; identity when signs is None."""
    x = np.asarray(x, dtype=np.float32)
    if signs is None:
        return x.copy()
    return bf16_round(rht_forward(x, signs))


def write_int4(key, value, slot_mapping, signs, k_cache, v_cache, k_scale, v_scale):
    """reshape_and_cache_int4 into numpy caches, in place.

    key, value: [T, Hk, D] float32 holding bf16 values.
    slot_mapping: [T] int64, entries < 0 are skipped.
    k_cache, v_cache: [num_blocks, block_size, Hk, D // 2] uint8.
    k_scale, v_scale: [num_blocks, block_size, Hk] uint32 (fp32 scale words).
    signs: [D] +-1 float32, or None to store the vectors unrotated.
    """
    slots = np.asarray(slot_mapping, dtype=np.int64)
    live = np.nonzero(slots >= 0)[0]
    if live.size == 0:
        return
    bs = k_cache.shape[1]
    blk = slots[live] // bs
    off = slots[live] % bs
    for src, cache, scales in ((key, k_cache, k_scale), (value, v_cache, v_scale)):
        r = rotate_to_bf16(np.asarray(src)[live], signs)
        q, word = quantize_int4(r)
        cache[blk, off] = pack_nibbles(q)
        scales[blk, off] = word


def gather_rows(pool, bt_row, L):
    """Rows of sequence positions 0..L-1: page bt_row[n // bs], row n % bs."""
    bs = pool.shape[1]
    n = np.arange(L)
    return pool[np.asarray(bt_row, dtype=np.int64)[n // bs], n % bs]


def _head_attention(q_rows, K, V, sm, pos=None, qpos=None, softcap=0.0, slopes=None, keep=None):
    """float64 softmax(S) v for q_rows [G, D], K/V [n, D]; returns ([G, D], lse [G]).

    S = sm * q.k, then, in the order of unified_attention_int4's tile loop: the soft cap
    S = softcap * tanh(S / softcap) when softcap > 0 (USE_SOFTCAP), the key mask (keep), and the
    ALiBi bias S += slope_g * (pos - qpos) (USE_ALIBI_SLOPES; pos = key positions, qpos = the
    query's position). A fully masked range returns o = 0, lse = -inf.
    """
    s = sm * (q_rows[:, None, :] * K[None, :, :]).sum(axis=-1)
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    if keep is not None:
        s = np.where(keep[None, :], s, -np.inf)
    if slopes is not None:
        s = s + np.asarray(slopes, np.float64)[:, None] * (np.asarray(pos, np.float64) - qpos)[None, :]
    m = s.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        return np.zeros((q_rows.shape[0], V.shape[1])), np.full(q_rows.shape[0], -np.inf)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e[:, :, None] * V[None, :, :]).sum(axis=1) / l
    return o, (m + np.log(l))[:, 0]


def decode_int4(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                signs, softmax_scale, num_splits=None, batch_index=None,
                window=0, softcap=0.0, sinks=None, alibi_slopes=None, q_len=1, return_lse=False,
                query_start_loc=None):
    """Paged decode attention over the INT4 cache (unified_attention_int4 semantics).

    q: [B, Hq, D] float32 holding bf16 values. Returns float64 [B, Hq, D] (rows of
    empty sequences are zero). With num_splits=S the kept keys of each sequence are cut
    into S ranges of ceil(n / S) positions (triton_turboquant_decode.py,
    _tq_decode_stage1 split range), each range is attended separately and the
    partial results are combined by the log-sum-exp merge (lse_merge); without it
    one softmax covers the whole sequence. batch_index restricts the work to some
    sequences (other rows are left zero).

    Score modifiers (unified_attention_int4 flags; the query is the token at position L - 1):
      window > 0      SLIDING_WINDOW: keys at positions n with (L - 1) - n < window are kept;
      softcap > 0     USE_SOFTCAP: S = softcap * tanh(S / softcap) on the scaled score;
      alibi_slopes    USE_ALIBI_SLOPES: [Hq] slopes, S += slope * (n - (L - 1));
      sinks           USE_SINKS: [Hq] logits that join each head's softmax denominator with no
                      value (the softmax state starts at M = sink, L = 1).

    Multi-token decode (unified_attention_int4 with max_seqlen_q > 1): sequence b has q_b query
    tokens, rows query_start_loc[b] .. query_start_loc[b + 1] - 1 of q (the varlen cu_seqlens_q
    layout; q_len = Q > 1 without it means q_b = Q for every b, rows b * Q + i). Query token i of
    sequence b sits at position L - q_b + i and attends causally to keys n <= L - q_b + i, every
    score modifier taken relative to its own position; the output has q's row layout. Sequences
    need L >= q_b.

    return_lse: also return the log-sum-exp of each row's scores, ln(sum_n e^{S_n}) (plus e^{sink}
    with sinks; -inf for a row with no key), float64 [rows, Hq] -- what
    triton_turboquant_decode_attention returns in lse_buf next to the output, so that a caller
    can merge this result with attention over other keys.
    """
    if q_len > 1 or query_start_loc is not None:
        q = np.asarray(q, dtype=np.float32)
        BQ, Hq, D = q.shape
        if query_start_loc is None:
            assert BQ % q_len == 0
            qsl = np.arange(0, BQ + 1, q_len)
        else:
            qsl = np.asarray(query_start_loc, dtype=np.int64)
        B = len(qsl) - 1
        out = np.zeros((BQ, Hq, D), dtype=np.float64)
        lse = np.full((BQ, Hq), -np.inf)
        if sinks is not None:
            lse[:] = np.asarray(sinks, np.float64)[None, :]   # a row with no key: the sink alone
        rows = range(B) if batch_index is None else batch_index
        for b in rows:
            L, qb = int(seq_lens[b]), int(qsl[b + 1] - qsl[b])
            for i in range(qb):
                r = int(qsl[b]) + i
                Li = L - qb + i + 1   # keys 0 .. L - q_b + i: the query at position Li - 1
                if Li <= 0:
                    continue
                o, l = decode_int4(q[r][None], k_cache, v_cache, k_scale, v_scale,
                                   np.asarray(block_table)[b][None], np.array([Li]), signs,
                                   softmax_scale, num_splits=num_splits, window=window, softcap=softcap,
                                   sinks=sinks, alibi_slopes=alibi_slopes, return_lse=True)
                out[r], lse[r] = o[0], l[0]
        return (out, lse) if return_lse else out
    q = np.asarray(q, dtype=np.float32)
    B, Hq, D = q.shape
    Hk = k_cache.shape[2]
    G = Hq // Hk
    q_rot = rotate_to_bf16(q, signs).astype(np.float64)
    sm = softmax_scale / D if signs is not None else softmax_scale
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse_out = np.full((B, Hq), -np.inf)
    if sinks is not None:
        lse_out[:] = np.asarray(sinks, np.float64)[None, :]   # a row with no key: the sink alone
    rows = range(B) if batch_index is None else batch_index
    for b in rows:
        L = int(seq_lens[b])
        if L == 0:
            continue
        lo = max(0, L - window) if window > 0 else 0   # first kept key
        K = dequant_int4(gather_rows(k_cache, block_table[b], L), gather_rows(k_scale, block_table[b], L))
        V = dequant_int4(gather_rows(v_cache, block_table[b], L), gather_rows(v_scale, block_table[b], L))
        pos = np.arange(L)
        keep = pos >= lo
        for h in range(Hk):
            qg = q_rot[b, h * G:(h + 1) * G]
            sl = None if alibi_slopes is None else np.asarray(alibi_slopes, np.float64)[h * G:(h + 1) * G]
            kw = dict(qpos=L - 1, softcap=softcap, slopes=sl)
            if num_splits is None:
                o, lse = _head_attention(qg, K[:, h], V[:, h], sm, pos=pos, keep=keep, **kw)
                parts = [(o, lse)]
            else:
                parts = []
                span = -(-(L - lo) // num_splits)
                for s in range(num_splits):
                    a, e = lo + s * span, min(lo + (s + 1) * span, L)
                    if a >= e:
                        continue
                    parts.append(_head_attention(qg, K[a:e, h], V[a:e, h], sm, pos=pos[a:e], **kw))
            if sinks is not None:
                parts.append((np.zeros((G, D)), np.asarray(sinks, np.float64)[h * G:(h + 1) * G]))
            if len(parts) == 1:
                o, lse = parts[0]
            else:
                o, lse = lse_merge([p[0] for p in parts], [p[1] for p in parts], return_lse=True)
            if signs is not None:
                o = rht_inverse_f64(o, signs) / D
            out[b, h * G:(h + 1) * G] = o
            lse_out[b, h * G:(h + 1) * G] = lse
    return (out, lse_out) if return_lse else out


def lse_merge(outs, lses, return_lse=False):
    """Combine per-split (o_s, lse_s): sum_s e^(lse_s - M) o_s / sum_s e^(lse_s - M), and (with
    return_lse) the merged log-sum-exp M + ln sum_s e^(lse_s - M).

    The stage-2 reduction itself is not on the pages (triton_turboquant_decode.py
    imports _fwd_kernel_stage2; int4_per_token_head.py imports reduce_segments);
    this is the standard max-shifted log-sum-exp combination of the partials that
    _tq_decode_stage1 stores (o = acc / l, lse = m + log l).
    """
    lses = np.stack([np.asarray(x, dtype=np.float64) for x in lses])     # [S, G]
    outs = np.stack([np.asarray(x, dtype=np.float64) for x in outs])     # [S, G, D]
    M = lses.max(axis=0)
    w = np.exp(lses - M)
    o = (w[:, :, None] * outs).sum(axis=0) / w.sum(axis=0)[:, None]
    return (o, M + np.log(w.sum(axis=0))) if return_lse else o
