"""Pins for the oracle's INT4 decode attention (oracle/int4_cache.py, decode_int4).

The reference points are torch's scaled_dot_product_attention in float64 (a library
routine), the explicit Sylvester matrix, and special cases with closed-form answers.
Identity used: with x~ = H(x^) * d1 / D for every rotated vector x^, the rotated-domain
attention softmax(scale / D * q_rot . k^) v^ mapped back by H(.) * d1 / D equals plain
attention softmax(scale * q~ . k~) v~ (H H = D I and d1 * d1 = 1).
"""

import numpy as np
import pytest
import torch

from oracle import hadamard, int4_cache
from quantized_paged_kv_int4_gb300 import workloads


def _build(case, num_blocks=None, signs=True, k=None, v=None):
    bt, nb = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=num_blocks, unused_fill=-1)
    seq, pos, slots = workloads.all_token_slots(bt, case.seq_lens)
    T = slots.numel()
    if k is None:
        k, v = workloads.kv_vectors(case, T)
    Hk, D = case.Hk, case.D
    kc = np.zeros((nb, 16, Hk, D // 2), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nb, 16, Hk), np.uint32)
    vs = np.zeros_like(ks)
    sg = workloads.rht_signs(D).numpy() if signs else None
    int4_cache.write_int4(workloads.to_numpy_f32(k), workloads.to_numpy_f32(v), slots.numpy(), sg,
                          kc, vc, ks, vs)
    q = workloads.to_numpy_f32(workloads.query(case))
    return dict(q=q, kc=kc, vc=vc, ks=ks, vs=vs, bt=bt.numpy(), lens=np.array(case.seq_lens), signs=sg)


def _run(c, scale, **kw):
    return int4_cache.decode_int4(c["q"], c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["lens"],
                                  c["signs"], scale, **kw)


def _unrotate(x, signs, D):
    """x~ = H x * d1 / D with the explicit matrix (float64)."""
    if signs is None:
        return np.asarray(x, np.float64)
    return (np.asarray(x, np.float64) @ hadamard.sylvester(D).T) * signs.astype(np.float64) / D


def _sdpa_expected(c, scale, Hq, Hk, D):
    G = Hq // Hk
    q_rot = int4_cache.rotate_to_bf16(c["q"], c["signs"])
    out = np.zeros(c["q"].shape, np.float64)
    for b, L in enumerate(c["lens"]):
        if L == 0:
            continue
        Kt = np.zeros((L, Hk, D))
        Vt = np.zeros((L, Hk, D))
        for n in range(L):  # position by position through the block table
            page, row = c["bt"][b, n // 16], n % 16
            Kt[n] = _unrotate(int4_cache.dequant_int4(c["kc"][page, row], c["ks"][page, row]), c["signs"], D)
            Vt[n] = _unrotate(int4_cache.dequant_int4(c["vc"][page, row], c["vs"][page, row]), c["signs"], D)
        qt = _unrotate(q_rot[b], c["signs"], D)                       # [Hq, D]
        Q = torch.from_numpy(qt)[None]                                 # [1, Hq, D] -> one query per head
        K = torch.from_numpy(Kt).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        V = torch.from_numpy(Vt).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(Q[:, :, None, :], K, V, scale=scale)
        out[b] = o[0, :, 0, :].numpy()
    return out


def test_decode_matches_sdpa_on_dequantized_cache():
    case = workloads.tiny_int4()
    c = _build(case, num_blocks=16)
    scale = 1.0 / np.sqrt(case.D)
    got = _run(c, scale)
    exp = _sdpa_expected(c, scale, case.Hq, case.Hk, case.D)
    assert np.max(np.abs(got - exp)) < 1e-12


def test_decode_gqa8_d128_matches_sdpa():
    case = workloads.DecodeCase("g8", 3, 16, 2, 128, [1, 17, 70], seed=3, outlier_channels=4)
    c = _build(case)
    scale = 1.0 / np.sqrt(case.D)
    assert np.max(np.abs(_run(c, scale) - _sdpa_expected(c, scale, 16, 2, 128))) < 1e-12


@pytest.mark.parametrize("S", [1, 2, 3, 4, 7, 16, 64, 200])
def test_split_lse_merge_equals_single_pass(S):
    case = workloads.tiny_int4(seed=4)
    c = _build(case, num_blocks=12)
    scale = 1.0 / np.sqrt(case.D)
    assert np.max(np.abs(_run(c, scale, num_splits=S) - _run(c, scale))) < 1e-12


def test_single_token_returns_its_value():
    case = workloads.DecodeCase("one", 2, 4, 2, 64, [1, 1], seed=5)
    c = _build(case)
    got = _run(c, 0.125)
    for b in range(2):
        page = c["bt"][b, 0]
        for hq in range(4):
            v = int4_cache.dequant_int4(c["vc"][page, 0, hq // 2], c["vs"][page, 0, hq // 2])
            assert np.max(np.abs(got[b, hq] - _unrotate(v, c["signs"], 64))) < 1e-12


def test_zero_query_is_uniform_mean_and_empty_sequence_is_zero():
    case = workloads.DecodeCase("zq", 3, 4, 2, 64, [33, 0, 5], seed=6)
    c = _build(case)
    c["q"][:] = 0.0
    got = _run(c, 0.3)
    assert np.all(got[1] == 0.0)
    for b in (0, 2):
        L = c["lens"][b]
        for hq in range(4):
            vs = [int4_cache.dequant_int4(c["vc"][c["bt"][b, n // 16], n % 16, hq // 2],
                                          c["vs"][c["bt"][b, n // 16], n % 16, hq // 2]) for n in range(L)]
            mean = _unrotate(np.mean(vs, axis=0), c["signs"], 64)
            assert np.max(np.abs(got[b, hq] - mean)) < 1e-12


def test_identical_keys_give_uniform_mean():
    case = workloads.DecodeCase("same", 1, 2, 1, 64, [40], seed=7)
    T = 40
    k, v = workloads.kv_vectors(case, T)
    k[:] = k[0]
    c = _build(case, k=k, v=v)
    got = _run(c, 0.5)
    vs = [int4_cache.dequant_int4(c["vc"][c["bt"][0, n // 16], n % 16, 0], c["vs"][c["bt"][0, n // 16], n % 16, 0])
          for n in range(T)]
    mean = _unrotate(np.mean(vs, axis=0), c["signs"], 64)
    assert np.max(np.abs(got[0] - mean)) < 1e-12


def test_unrotated_exactly_representable_cache_is_textbook_attention():
    # rows on the grid (n - 8) / 4 with both ends present: scale 0.25, zp 8, every value exact in INT4
    case = workloads.DecodeCase("exact", 2, 6, 3, 64, [29, 50], seed=8)
    rng = np.random.default_rng(8)
    T = sum(case.seq_lens)

    def grid():
        n = rng.integers(0, 16, size=(T, 3, 64))
        n[..., 0] = 0
        n[..., 1] = 15
        return torch.from_numpy((n - 8) / 4.0).to(torch.bfloat16)

    k, v = grid(), grid()
    c = _build(case, signs=False, k=k, v=v)
    got = _run(c, 0.2)
    # the gather order equals the generation order: sequence b's tokens are contiguous in k, v
    off = 0
    for b, L in enumerate(case.seq_lens):
        Q = torch.from_numpy(c["q"][b].astype(np.float64))[None, :, None, :]
        K = k[off:off + L].to(torch.float64).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
        V = v[off:off + L].to(torch.float64).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=0.2)[0, :, 0, :].numpy()
        assert np.max(np.abs(got[b] - o)) < 1e-12
        off += L


@pytest.mark.parametrize("Q", [2, 4])
def test_multi_token_decode_matches_causal_sdpa(Q):
    """Q query tokens per sequence at positions L - Q .. L - 1, each attending causally: float64 SDPA
    with an explicit boolean causal mask on the dequantized cache."""
    case = workloads.DecodeCase("mtok", 3, 4 * Q, 2, 64, [5, 40, 17], seed=40 + Q)
    c = _build(case)
    B, Hq, D = 3, 4, 64
    G = Hq // 2
    rng = np.random.default_rng(Q)
    q = int4_cache.bf16_round(rng.standard_normal((B * Q, Hq, D)).astype(np.float32))
    scale = 1.0 / np.sqrt(D)
    got = int4_cache.decode_int4(q, c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["lens"], c["signs"], scale,
                                 q_len=Q)
    q_rot = int4_cache.rotate_to_bf16(q, c["signs"])
    for b, L in enumerate(c["lens"]):
        Kt = np.zeros((L, 2, D)); Vt = np.zeros((L, 2, D))
        for n in range(L):
            page, row = c["bt"][b, n // 16], n % 16
            Kt[n] = _unrotate(int4_cache.dequant_int4(c["kc"][page, row], c["ks"][page, row]), c["signs"], D)
            Vt[n] = _unrotate(int4_cache.dequant_int4(c["vc"][page, row], c["vs"][page, row]), c["signs"], D)
        Qm = torch.from_numpy(np.stack([_unrotate(q_rot[b * Q + i], c["signs"], D) for i in range(Q)], axis=1))  # [Hq, Q, D]
        K = torch.from_numpy(np.repeat(Kt.transpose(1, 0, 2), G, axis=0))
        V = torch.from_numpy(np.repeat(Vt.transpose(1, 0, 2), G, axis=0))
        allowed = torch.from_numpy(np.arange(L)[None, :] <= (L - Q + np.arange(Q))[:, None])  # [Q, L]
        o = torch.nn.functional.scaled_dot_product_attention(Qm, K, V, attn_mask=allowed, scale=scale)  # [Hq, Q, D]
        for i in range(Q):
            assert np.max(np.abs(got[b * Q + i] - o[:, i].numpy())) < 1e-12


# ---------------------------------------------------------------------------------------------
# The merged log-sum-exp (return_lse): closed forms and split invariance
# ---------------------------------------------------------------------------------------------
def test_lse_of_a_zero_query_is_the_log_of_the_length():
    """Every score is 0, so ln(sum_n e^0) = ln L exactly; with a sink s: ln(L + e^s); an empty row:
    -inf without a sink, s with one."""
    case = workloads.DecodeCase("zl", 3, 4, 2, 64, [33, 0, 5], seed=21)
    c = _build(case)
    c["q"][:] = 0.0
    _, lse = _run(c, 0.3, return_lse=True)
    assert np.allclose(lse[0], np.log(33.0), rtol=0, atol=1e-12) and np.allclose(lse[2], np.log(5.0), atol=1e-12)
    assert np.all(lse[1] == -np.inf)
    sinks = np.array([0.5, -1.0, 2.0, 0.0])
    for S in (None, 3):
        _, lse = _run(c, 0.3, return_lse=True, sinks=sinks, num_splits=S)
        assert np.allclose(lse[0], np.log(33.0 + np.exp(sinks)), atol=1e-12)
        assert np.allclose(lse[1], sinks, atol=0)


def test_lse_of_identical_keys_grows_by_log_length():
    """L copies of one key: lse(L) - lse(1) = ln L (each copy adds the same e^S)."""
    case = workloads.DecodeCase("same", 1, 2, 1, 64, [40], seed=22)
    k, v = workloads.kv_vectors(case, 40)
    k[:] = k[0]
    c = _build(case, k=k, v=v)
    _, lse40 = _run(c, 0.5, return_lse=True)
    c["lens"] = np.array([1])
    _, lse1 = _run(c, 0.5, return_lse=True)
    assert np.max(np.abs(lse40 - lse1 - np.log(40.0))) < 1e-12


@pytest.mark.parametrize("S", [1, 2, 3, 7, 64])
def test_lse_of_split_merge_equals_single_pass(S):
    case = workloads.tiny_int4(seed=23)
    c = _build(case, num_blocks=12)
    o1, l1 = _run(c, 0.125, return_lse=True)
    oS, lS = _run(c, 0.125, return_lse=True, num_splits=S)
    assert np.max(np.abs(lS - l1)) < 1e-12 and np.max(np.abs(oS - o1)) < 1e-12


def test_lse_multi_token_rows_are_their_prefix_lse():
    """Query token i of a Q-token row sees keys 0 .. L - Q + i: its lse is the single-token lse
    over that prefix."""
    case = workloads.DecodeCase("mt", 2, 4, 2, 64, [30, 45], seed=24)
    c = _build(case)
    Q = 3
    q = np.repeat(c["q"], Q, axis=0)
    _, lse = int4_cache.decode_int4(q, c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["lens"], c["signs"], 0.2,
                                    q_len=Q, return_lse=True)
    for b in range(2):
        for i in range(Q):
            Li = c["lens"][b] - Q + i + 1
            _, one = int4_cache.decode_int4(c["q"][b][None], c["kc"], c["vc"], c["ks"], c["vs"], c["bt"][b][None],
                                            np.array([Li]), c["signs"], 0.2, return_lse=True)
            assert np.max(np.abs(lse[b * Q + i] - one[0])) < 1e-12


@pytest.mark.parametrize("window", [0, 6])
def test_ragged_multi_query_with_window_and_alibi_matches_masked_sdpa(window):
    """Ragged query counts (query_start_loc, the varlen cu_seqlens_q layout): sequence b's q_b tokens
    sit at positions L - q_b .. L - 1; token at position p sees keys n <= p (and p - n < window),
    with the ALiBi bias slope * (n - p). Expected: float64 SDPA with that additive float mask."""
    lens = [9, 40, 17, 3]
    counts = [3, 0, 5, 1]
    case = workloads.DecodeCase("rag", 4, 4, 2, 64, lens, seed=50 + window)
    c = _build(case)
    Hq, D, G = 4, 64, 2
    qsl = np.concatenate([[0], np.cumsum(counts)])
    rng = np.random.default_rng(window)
    q = int4_cache.bf16_round(rng.standard_normal((qsl[-1], Hq, D)).astype(np.float32))
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])
    scale = 1.0 / np.sqrt(D)
    got = int4_cache.decode_int4(q, c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["lens"], c["signs"], scale,
                                 query_start_loc=qsl, window=window, alibi_slopes=slopes)
    q_rot = int4_cache.rotate_to_bf16(q, c["signs"])
    for b, L in enumerate(lens):
        qb = counts[b]
        if qb == 0:
            continue
        Kt = np.zeros((L, 2, D)); Vt = np.zeros((L, 2, D))
        for n in range(L):
            page, row = c["bt"][b, n // 16], n % 16
            Kt[n] = _unrotate(int4_cache.dequant_int4(c["kc"][page, row], c["ks"][page, row]), c["signs"], D)
            Vt[n] = _unrotate(int4_cache.dequant_int4(c["vc"][page, row], c["vs"][page, row]), c["signs"], D)
        rows = range(qsl[b], qsl[b + 1])
        Qm = torch.from_numpy(np.stack([_unrotate(q_rot[r], c["signs"], D) for r in rows], axis=1))  # [Hq, qb, D]
        K = torch.from_numpy(np.repeat(Kt.transpose(1, 0, 2), G, axis=0))
        V = torch.from_numpy(np.repeat(Vt.transpose(1, 0, 2), G, axis=0))
        pos = L - qb + np.arange(qb)                       # query positions
        n = np.arange(L)
        keep = n[None, :] <= pos[:, None]
        if window:
            keep &= (pos[:, None] - n[None, :]) < window
        bias = slopes[:, None, None] * (n[None, None, :] - pos[None, :, None])   # [Hq, qb, L]
        mask = torch.from_numpy(np.where(keep[None], bias, -np.inf))
        o = torch.nn.functional.scaled_dot_product_attention(Qm, K, V, attn_mask=mask, scale=scale)
        for i, r in enumerate(rows):
            assert np.max(np.abs(got[r] - o[:, i].numpy())) < 1e-12


def test_uniform_query_counts_equal_the_q_len_layout():
    case = workloads.DecodeCase("u", 3, 4, 2, 64, [20, 33, 7], seed=55)
    c = _build(case)
    rng = np.random.default_rng(3)
    q = int4_cache.bf16_round(rng.standard_normal((9, 4, 64)).astype(np.float32))
    a = int4_cache.decode_int4(q, c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["lens"], c["signs"], 0.1, q_len=3)
    b = int4_cache.decode_int4(q, c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["lens"], c["signs"], 0.1,
                               query_start_loc=np.array([0, 3, 6, 9]))
    assert np.array_equal(a, b)
