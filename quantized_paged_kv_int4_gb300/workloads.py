"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random tensors and lays them out (paged block tables,
slot mappings, synthetic cache bytes). It performs none of the method's
arithmetic: no rotation, no quantization, no attention.

Seeding: tensor k of a case is drawn from ``torch.Generator().manual_seed(seed + k)``
(k = 1 q, 2 K, 3 V, 4 block-table permutation, 5 sequence lengths, 6 slot mapping,
7 outlier channels, 8 cache bytes, 9 slot-mapping holes).

The random-sign vector of the Hadamard rotation is generated the way
int4_per_token_head.py, _get_rht_signs does: a CPU torch generator seeded with
0x9E3779B9 + round * 0x517CC1B7 and 2 * bernoulli(0.5) - 1.
"""

from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16


def _gen(seed, k):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + int(k))
    return g


def rht_signs(D, round_idx=0):
    """float32 [D] of +-1 (int4_per_token_head.py, _get_rht_signs)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(0x9E3779B9 + round_idx * 0x517CC1B7)
    return 2.0 * torch.bernoulli(torch.full((D,), 0.5), generator=g) - 1.0


# ----------------------------------------------------------------------------
# configurations (the five workloads of the hot path)
# ----------------------------------------------------------------------------


@dataclass
class DecodeCase:
    name: str
    B: int
    Hq: int
    Hk: int
    D: int
    seq_lens: list
    num_splits: int = 0          # 0: library heuristic
    block_size: int = BLOCK_SIZE
    outlier_channels: int = 0    # channels of K scaled by outlier_scale before rotation
    outlier_scale: float = 10.0
    pool_bytes: int = 0          # if set, the page pool is this large (pages scattered in it)
    seed: int = 0
    extra: dict = field(default_factory=dict)


def tiny_int4(seed=0):
    """B=2, Hq=4, Hk=2, D=64, block 16, seq_lens {37, 100}, 4 KV splits."""
    return DecodeCase("tiny_int4", 2, 4, 2, 64, [37, 100], num_splits=4, seed=seed)


def llama8b_int4(seed=0):
    """B=32, Hq=32, Hk=8, D=128, seq_lens uniform in [1024, 8192], K with 4 x10 outlier channels."""
    g = _gen(seed, 5)
    lens = torch.randint(1024, 8193, (32,), generator=g).tolist()
    return DecodeCase("llama3_8b_int4", 32, 32, 8, 128, lens, num_splits=0,
                      outlier_channels=4, seed=seed)


def long_context_int4(seed=0):
    """B=4, Hq=64, Hk=8, D=128, seq_len 131072 each, 64 KV splits, pages in a 40 GB pool."""
    return DecodeCase("long_context_int4", 4, 64, 8, 128, [131072] * 4, num_splits=64,
                      pool_bytes=40_000_000_000, seed=seed)


def turboquant_fp8(value_bits=4, seed=0):
    """B=64, Hq=32, Hk=8, D=128, seq_len 4096, FP8 keys + 4-bit (or 3-bit) values."""
    return DecodeCase("turboquant_fp8_v%d" % value_bits, 64, 32, 8, 128, [4096] * 64,
                      num_splits=0, seed=seed, extra={"value_bits": value_bits})


def turboquant_mse(key_bits=3, value_bits=4, seed=0):
    """B=64, Hq=32, Hk=8, D=128, seq_len 4096, MSE keys (key_bits-bit centroid indices + fp16
    norm) + 4-bit (or 3-bit) values."""
    return DecodeCase("turboquant_mse_k%dv%d" % (key_bits, value_bits), 64, 32, 8, 128, [4096] * 64,
                      num_splits=0, seed=seed, extra={"key_bits": key_bits, "value_bits": value_bits})


# ----------------------------------------------------------------------------
# paged layout
# ----------------------------------------------------------------------------


def pages_needed(seq_lens, block_size=BLOCK_SIZE):
    return [-(-int(L) // block_size) for L in seq_lens]


def paged_layout(seq_lens, seed, block_size=BLOCK_SIZE, num_blocks=None, unused_fill=0):
    """Random physical placement of every sequence's pages.

    Returns (block_table int32 [B, max_blocks], num_blocks). The physical pages of
    all sequences are a random subset (a random permutation when num_blocks is
    the exact number needed) of range(num_blocks); entries past a sequence's
    last page hold unused_fill.
    """
    need = pages_needed(seq_lens, block_size)
    total = sum(need)
    if num_blocks is None:
        num_blocks = max(total, 1)
    assert num_blocks >= total
    g = _gen(seed, 4)
    if num_blocks == total:
        phys = torch.randperm(num_blocks, generator=g)[:total]
    else:
        # a random subset of a large pool without materialising a full permutation
        chosen = set()
        picks = []
        while len(picks) < total:
            cand = torch.randint(0, num_blocks, (2 * (total - len(picks)) + 16,), generator=g).tolist()
            for c in cand:
                if c not in chosen:
                    chosen.add(c)
                    picks.append(c)
                    if len(picks) == total:
                        break
        phys = torch.tensor(picks, dtype=torch.int64)
    max_blocks = max(max(need), 1)
    bt = torch.full((len(seq_lens), max_blocks), unused_fill, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = phys[pos:pos + n].to(torch.int32)
        pos += n
    return bt, num_blocks


def slots_for_positions(block_table, seq_index, positions, block_size=BLOCK_SIZE):
    """Flat cache slots (int64) of sequence positions: page * block_size + row."""
    bt = block_table.to(torch.int64)
    pos = torch.as_tensor(positions, dtype=torch.int64)
    b = torch.as_tensor(seq_index, dtype=torch.int64)
    return bt[b, pos // block_size] * block_size + pos % block_size


def all_token_slots(block_table, seq_lens, block_size=BLOCK_SIZE):
    """(seq_index, position, slot) for every token of every sequence, concatenated."""
    seq = torch.cat([torch.full((int(L),), b, dtype=torch.int64) for b, L in enumerate(seq_lens)])
    pos = torch.cat([torch.arange(int(L), dtype=torch.int64) for L in seq_lens])
    return seq, pos, slots_for_positions(block_table, seq, pos, block_size)


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------


def bf16_normal(shape, seed, k, device="cpu"):
    """N(0, 1) drawn in fp32 from the seeded CPU generator, stored as bf16."""
    x = torch.randn(shape, generator=_gen(seed, k), dtype=torch.float32)
    return x.to(torch.bfloat16).to(device)


def outlier_channels(D, n, seed):
    if n == 0:
        return torch.zeros((0,), dtype=torch.int64)
    return torch.randperm(D, generator=_gen(seed, 7))[:n]


def kv_vectors(case, T):
    """K and V [T, Hk, D] bf16 for T tokens; K gets the case's outlier channels."""
    k = torch.randn((T, case.Hk, case.D), generator=_gen(case.seed, 2), dtype=torch.float32)
    ch = outlier_channels(case.D, case.outlier_channels, case.seed)
    if ch.numel():
        k[:, :, ch] *= case.outlier_scale
    v = torch.randn((T, case.Hk, case.D), generator=_gen(case.seed, 3), dtype=torch.float32)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def query(case, dtype=torch.bfloat16):
    q = torch.randn((case.B, case.Hq, case.D), generator=_gen(case.seed, 1), dtype=torch.float32)
    return q.to(dtype)


def write_case(T=16384, Hk=8, D=128, hole_frac=0.05, seed=0, num_blocks=None):
    """Cache-write workload: T new tokens, slot_mapping a permutation of pool slots with holes.

    Returns (key, value, slot_mapping int64 [T], num_blocks).
    """
    if num_blocks is None:
        num_blocks = -(-T // BLOCK_SIZE) + 8
    perm = torch.randperm(num_blocks * BLOCK_SIZE, generator=_gen(seed, 6))[:T]
    holes = torch.rand((T,), generator=_gen(seed, 9)) < hole_frac
    slots = torch.where(holes, torch.full_like(perm, -1), perm).to(torch.int64)
    k = torch.randn((T, Hk, D), generator=_gen(seed, 2), dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((T, Hk, D), generator=_gen(seed, 3), dtype=torch.float32).to(torch.bfloat16)
    return k, v, slots, num_blocks


def fwht_rows(rows=65536, seed=0):
    return torch.randn((rows, 128), generator=_gen(seed, 1), dtype=torch.float32).to(torch.bfloat16)


# ----------------------------------------------------------------------------
# synthetic cache bytes (inputs for the read side when no write precedes it)
# ----------------------------------------------------------------------------


def random_int4_pages(num_pages, Hk, D, seed, device="cpu", generator=None):
    """Random packed nibble pages and scale words for num_pages pages.

    Returns (k_bytes, v_bytes) uint8 [num_pages, 16, Hk, D // 2] and
    (k_words, v_words) int32 [num_pages, 16, Hk] whose fp32 reading is a positive
    scale in [1/8, 1/2) with a random 4-bit value in the low mantissa bits.
    """
    g = generator if generator is not None else _gen(seed, 8)
    dev = "cpu" if generator is None else device
    shape = (num_pages, BLOCK_SIZE, Hk)
    kb = torch.randint(0, 256, shape + (D // 2,), generator=g, dtype=torch.uint8, device=dev)
    vb = torch.randint(0, 256, shape + (D // 2,), generator=g, dtype=torch.uint8, device=dev)

    def words():
        mant = torch.randint(0, 1 << 23, shape, generator=g, dtype=torch.int32, device=dev)
        expo = torch.randint(124, 126, shape, generator=g, dtype=torch.int32, device=dev)
        return (expo << 23) | mant

    kw, vw = words(), words()
    return kb.to(device), vb.to(device), kw.to(device), vw.to(device)


def turboquant_slot_bytes(D, value_bits):
    """FP8 key (D bytes) + ceil(D * bits / 8) value bytes + fp16 scale + fp16 zero, padded to 16."""
    raw = D + (-(-D * value_bits // 8)) + 4
    return -(-raw // 16) * 16


def random_turboquant_slots(n_slots_shape, D, value_bits, seed, k=None, v=None):
    """Synthetic combined slots [..., slot_bytes] uint8.

    Keys: torch's float8_e4m3fn cast of N(0, 1) draws (or of k). Values: per slot a
    min/max uniform grid -- zero = min, scale = (max - min) / (2^bits - 1), both
    float16, indices round((v - zero) / scale) clipped to the grid -- packed in the
    page's 4-bit (two per byte) or 3-bit (LSB-first stream) order. The writer is not
    part of the read path; this only produces valid cache bytes.
    """
    shape = tuple(n_slots_shape)
    if k is None:
        k = torch.randn(shape + (D,), generator=_gen(seed, 2), dtype=torch.float32)
    if v is None:
        v = torch.randn(shape + (D,), generator=_gen(seed, 3), dtype=torch.float32)
    kbytes = k.to(torch.float8_e4m3fn).view(torch.uint8)
    levels = (1 << value_bits) - 1
    vmin = v.min(dim=-1, keepdim=True).values
    vmax = v.max(dim=-1, keepdim=True).values
    zero = vmin.to(torch.float16)
    scale = ((vmax - vmin) / levels).clamp_min(1e-4).to(torch.float16)
    idx = torch.round((v - zero.float()) / scale.float()).clamp(0, levels).to(torch.int64)
    vdb = -(-D * value_bits // 8)
    vbytes = torch.zeros(shape + (vdb,), dtype=torch.int64)
    if value_bits == 4:
        vbytes = (idx[..., 0::2] | (idx[..., 1::2] << 4))
    else:
        for d in range(D):
            bit = 3 * d
            vbytes[..., bit // 8] |= (idx[..., d] << (bit % 8)) & 0xFF
            if bit % 8 > 5:
                vbytes[..., bit // 8 + 1] |= idx[..., d] >> (8 - bit % 8)
    sc = scale.view(torch.int16).to(torch.int64) & 0xFFFF
    zr = zero.view(torch.int16).to(torch.int64) & 0xFFFF
    sb = turboquant_slot_bytes(D, value_bits)
    out = torch.zeros(shape + (sb,), dtype=torch.uint8)
    out[..., :D] = kbytes
    out[..., D:D + vdb] = vbytes.to(torch.uint8)
    out[..., D + vdb] = (sc & 0xFF).to(torch.uint8)[..., 0]
    out[..., D + vdb + 1] = (sc >> 8).to(torch.uint8)[..., 0]
    out[..., D + vdb + 2] = (zr & 0xFF).to(torch.uint8)[..., 0]
    out[..., D + vdb + 3] = (zr >> 8).to(torch.uint8)[..., 0]
    return out


def to_numpy_f32(t):
    """float32 numpy copy of a (bf16/fp16/fp32) tensor."""
    return t.detach().to("cpu").to(torch.float32).numpy()


def as_u32(t):
    return np.ascontiguousarray(t.detach().to("cpu").view(torch.int32).numpy().view(np.uint32))


# ----------------------------------------------------------------------------
# TurboQuant MSE-key slots (synthetic codebook, rotation and cache bytes)
# ----------------------------------------------------------------------------


def turboquant_mse_layout(D, key_bits, value_bits):
    """(mse_bytes, key_packed_size, slot_bytes): key_bits-bit indices, the fp16 norm right after
    them (no QJL bytes), the values from key_packed_size = mse_bytes + 2, then fp16 scale and
    zero; the slot padded to a multiple of 16 bytes."""
    mse = -(-D * key_bits // 8)
    kps = mse + 2
    raw = kps + (-(-D * value_bits // 8)) + 4
    return mse, kps, -(-raw // 16) * 16


def mse_codebook(key_bits, D):
    """A synthetic centroid table [2^key_bits] float32: the N(0, 1/D) quantiles at the bin
    midpoints (j + 1/2) / 2^key_bits (no trained codebook is on the pages)."""
    n = 1 << key_bits
    p = (torch.arange(n, dtype=torch.float64) + 0.5) / n
    return (torch.special.ndtri(p) / np.sqrt(D)).to(torch.float32)


def random_rotation(D, seed):
    """A seeded random orthogonal [D, D] float32 matrix (QR of a Gaussian draw, signs fixed)."""
    a = torch.randn((D, D), generator=_gen(seed, 10), dtype=torch.float64)
    qm, r = torch.linalg.qr(a)
    return (qm * torch.sign(torch.diagonal(r))[None, :]).to(torch.float32).contiguous()


def _pack_lsb_stream(idx, bits, nbytes):
    """[..., D] indices -> [..., nbytes] LSB-first bit stream (index d at bit bits * d)."""
    out = torch.zeros(idx.shape[:-1] + (nbytes,), dtype=torch.int64)
    for d in range(idx.shape[-1]):
        bit = bits * d
        out[..., bit // 8] |= (idx[..., d] << (bit % 8)) & 0xFF
        if bit % 8 + bits > 8:
            out[..., bit // 8 + 1] |= idx[..., d] >> (8 - bit % 8)
    return out.to(torch.uint8)


def random_turboquant_mse_slots(n_slots_shape, D, key_bits, value_bits, seed):
    """Synthetic MSE-key slots [..., slot_bytes] uint8: uniform random key indices, fp16 norms
    |N(0, 1)| * sqrt(D) / 2 + 1, values as random_turboquant_slots (min/max grid)."""
    shape = tuple(n_slots_shape)
    mse, kps, sb = turboquant_mse_layout(D, key_bits, value_bits)
    idx = torch.randint(0, 1 << key_bits, shape + (D,), generator=_gen(seed, 2), dtype=torch.int64)
    norms = (torch.randn(shape, generator=_gen(seed, 11), dtype=torch.float32).abs() * (np.sqrt(D) / 2) + 1.0)
    nb = norms.to(torch.float16).view(torch.int16).to(torch.int64) & 0xFFFF
    fp8 = random_turboquant_slots(shape, D, value_bits, seed)          # reuse its value bytes
    vlen = -(-D * value_bits // 8) + 4
    out = torch.zeros(shape + (sb,), dtype=torch.uint8)
    out[..., :mse] = _pack_lsb_stream(idx, key_bits, mse)
    out[..., mse] = (nb & 0xFF).to(torch.uint8)
    out[..., mse + 1] = (nb >> 8).to(torch.uint8)
    out[..., kps:kps + vlen] = fp8[..., D:D + vlen]
    return out


# ----------------------------------------------------------------------------
# kpool compress-and-write inputs
# ----------------------------------------------------------------------------


def kpool_case(n_pools=16384, pool_size=4, page_size=64, seed=0, extra_blocks=4):
    """(slot_k bf16 [n, pool, 128], slot_score fp32 [n, pool, 128], ape fp32 [pool, 128], loc int64 [n],
    num_blocks): N(0, 1) keys, N(0, 4) scores, N(0, 1/4) position biases, locations a random
    permutation of the pool's slots."""
    num_blocks = -(-n_pools // page_size) + extra_blocks
    slot_k = torch.randn((n_pools, pool_size, 128), generator=_gen(seed, 2)).to(torch.bfloat16)
    slot_score = torch.randn((n_pools, pool_size, 128), generator=_gen(seed, 12)) * 2.0
    ape = torch.randn((pool_size, 128), generator=_gen(seed, 13)) * 0.5
    loc = torch.randperm(num_blocks * page_size, generator=_gen(seed, 6))[:n_pools].to(torch.int64)
    return slot_k, slot_score, ape, loc, num_blocks
