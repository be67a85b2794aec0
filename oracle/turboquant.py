"""Decode attention over the TurboQuant combined K+V slot (FP8 keys).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source page: triton_turboquant_decode.py, _tq_decode_stage1 with KEY_FP8=1 and
triton_turboquant_decode_attention. One slot per (page, row, kv-head) of
slot_bytes bytes:
  bytes [0, D)                  key, one FP8 E4M3FN code per dimension
                                (key_packed_size = D for FP8 keys)
  bytes [D, D + VDB)            value indices, VDB = ceil(D * bits / 8):
                                4-bit: dimension d in byte d // 2, low nibble when
                                d is even, high nibble when d is odd;
                                3-bit: LSB-first bit stream, index of d =
                                ((byte[o] | byte[o + 1] << 8) >> (3d mod 8)) & 7
                                with o = 3d // 8
  bytes [D + VDB, D + VDB + 2)  value scale, float16 little-endian
  bytes [D + VDB + 2, + 4)      value zero,  float16 little-endian
  rest                          padding
A value dequantizes to idx * scale + zero; the score is attn_scale * sum(q * k)
with q used as given (the FP8 path feeds the query straight in). Softmax and the
weighted sum are evaluated here in float64; the output keeps q's dtype (fp32).
"""

import numpy as np

from .formats import e4m3fn_to_f64, fp16_to_f64


def value_data_bytes(D, value_bits):
    """ceil(D * bits / 8) (triton_turboquant_decode.py, _get_layout)."""
    return -(-D * value_bits // 8)


def _bit_field(slots, start, D, bits):
    """Index of dimension d = ((byte[o] | byte[o + 1] << 8) >> (bits * d mod 8)) & (2^bits - 1) with
    o = start + bits * d // 8: the LSB-first stream the page reads for 3-bit values and MSE keys."""
    d = np.arange(D)
    o = start + (bits * d) // 8
    raw = slots[..., o].astype(np.int64) | (slots[..., o + 1].astype(np.int64) << 8)
    return (raw >> ((bits * d) % 8)) & ((1 << bits) - 1)


def dequant_values(slots, D, value_bits, voff):
    """Values (float64 [..., D]) of slot rows whose value data start at byte voff: idx * scale + zero."""
    slots = np.asarray(slots, dtype=np.uint8)
    vdb = value_data_bytes(D, value_bits)
    d = np.arange(D)
    if value_bits == 4:
        raw = slots[..., voff + d // 2].astype(np.int64)
        idx = (raw >> (4 * (d % 2))) & 0xF
    elif value_bits == 3:
        idx = _bit_field(slots, voff, D, 3)
    else:
        raise ValueError(value_bits)
    base = voff + vdb
    sc_bits = slots[..., base].astype(np.uint16) | (slots[..., base + 1].astype(np.uint16) << 8)
    zr_bits = slots[..., base + 2].astype(np.uint16) | (slots[..., base + 3].astype(np.uint16) << 8)
    return idx.astype(np.float64) * fp16_to_f64(sc_bits)[..., None] + fp16_to_f64(zr_bits)[..., None]


def dequant_slots(slots, D, value_bits):
    """Keys and values (float64 [..., D] each) of slot byte rows [..., slot_bytes]."""
    slots = np.asarray(slots, dtype=np.uint8)
    k = e4m3fn_to_f64(slots[..., :D])
    vdb = value_data_bytes(D, value_bits)
    d = np.arange(D)
    if value_bits == 4:
        raw = slots[..., D + d // 2].astype(np.int64)
        idx = (raw >> (4 * (d % 2))) & 0xF
    elif value_bits == 3:
        o = D + (3 * d) // 8
        raw = slots[..., o].astype(np.int64) | (slots[..., o + 1].astype(np.int64) << 8)
        idx = (raw >> ((3 * d) % 8)) & 0x7
    else:
        raise ValueError(value_bits)
    base = D + vdb
    sc_bits = slots[..., base].astype(np.uint16) | (slots[..., base + 1].astype(np.uint16) << 8)
    zr_bits = slots[..., base + 2].astype(np.uint16) | (slots[..., base + 3].astype(np.uint16) << 8)
    scale = fp16_to_f64(sc_bits)
    zero = fp16_to_f64(zr_bits)
    v = idx.astype(np.float64) * scale[..., None] + zero[..., None]
    return k, v


def decode_tq(q, kv_cache, value_bits, block_table, seq_lens, attn_scale, batch_index=None,
              return_lse=False):
    """q: [B, Hq, D] float32; kv_cache: [num_blocks, block_size, Hk, slot_bytes] uint8.

    Returns float64 [B, Hq, D]; rows of empty sequences are zero. return_lse: also the
    log-sum-exp ln(sum_n e^{score_n}) of each row, float64 [B, Hq] (-inf for an empty row), the
    lse_buf that triton_turboquant_decode_attention returns next to the output.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hk = kv_cache.shape[2]
    G = Hq // Hk
    bs = kv_cache.shape[1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf)
    rows = range(B) if batch_index is None else batch_index
    for b in rows:
        L = int(seq_lens[b])
        if L == 0:
            continue
        n = np.arange(L)
        slots = kv_cache[np.asarray(block_table[b], dtype=np.int64)[n // bs], n % bs]  # [L, Hk, slot]
        K, V = dequant_slots(slots, D, value_bits)
        for hq in range(Hq):
            h = hq // G
            s = attn_scale * (q[b, hq][None, :] * K[:, h, :]).sum(axis=-1)
            e = np.exp(s - s.max())
            out[b, hq] = (e[:, None] * V[:, h, :]).sum(axis=0) / e.sum()
            lse[b, hq] = s.max() + np.log(e.sum())
    return (out, lse) if return_lse else out


# ----------------------------------------------------------------------------------------------
# MSE keys (_tq_decode_stage1 with KEY_FP8 = 0; triton_turboquant_decode_attention, key_fp8=False)
# ----------------------------------------------------------------------------------------------


def mse_key_bytes(D, key_bits):
    """MSE_BYTES = ceil(D * mse_bits / 8) (_get_layout)."""
    return -(-D * key_bits // 8)


def dequant_mse_keys(slots, D, key_bits, centroids, norm_correction):
    """(c, norm) of slot rows: c [..., D] float64 the centroid vector of the key's indices
    (LSB-first key_bits-bit stream from byte 0), divided by sqrt(sum c^2 + 1e-16) when
    norm_correction (NORM_CORRECTION); norm [...] the float16 at byte MSE_BYTES."""
    slots = np.asarray(slots, dtype=np.uint8)
    idx = _bit_field(slots, 0, D, key_bits)
    c = np.asarray(centroids, dtype=np.float32).astype(np.float64)[idx]
    if norm_correction:
        c = c / np.sqrt((c * c).sum(axis=-1, keepdims=True) + 1e-16)
    mb = mse_key_bytes(D, key_bits)
    nbits = slots[..., mb].astype(np.uint16) | (slots[..., mb + 1].astype(np.uint16) << 8)
    return c, fp16_to_f64(nbits)


def decode_tq_mse(q, kv_cache, key_bits, key_packed_size, value_bits, centroids, norm_correction, Pi,
                  block_table, seq_lens, attn_scale, batch_index=None):
    """TurboQuant decode with MSE keys. q: [B, Hq, D] float32 (the original query); the score of
    key n is attn_scale * norm_n * (q_rot . c_n) with q_rot = q @ Pi^T (the launcher's GEMM);
    the values start at byte key_packed_size of the slot. Returns float64 [B, Hq, D]."""
    q = np.asarray(q, dtype=np.float32).astype(np.float64)
    B, Hq, D = q.shape
    q_rot = q @ np.asarray(Pi, dtype=np.float32).astype(np.float64).T
    Hk = kv_cache.shape[2]
    G = Hq // Hk
    bs = kv_cache.shape[1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rows = range(B) if batch_index is None else batch_index
    for b in rows:
        L = int(seq_lens[b])
        if L == 0:
            continue
        n = np.arange(L)
        slots = kv_cache[np.asarray(block_table[b], dtype=np.int64)[n // bs], n % bs]  # [L, Hk, slot]
        c, norm = dequant_mse_keys(slots, D, key_bits, centroids, norm_correction)
        V = dequant_values(slots, D, value_bits, key_packed_size)
        for hq in range(Hq):
            h = hq // G
            s = attn_scale * norm[:, h] * (q_rot[b, hq][None, :] * c[:, h, :]).sum(axis=-1)
            e = np.exp(s - s.max())
            out[b, hq] = (e[:, None] * V[:, h, :]).sum(axis=0) / e.sum()
    return out
