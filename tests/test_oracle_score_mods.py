"""Pins for the oracle's score modifiers on the INT4 decode (oracle/int4_cache.py, decode_int4:
sliding window, soft cap, ALiBi, attention sinks -- unified_attention_int4's SLIDING_WINDOW,
USE_SOFTCAP, USE_ALIBI_SLOPES and USE_SINKS).

Reference points: torch's scaled_dot_product_attention in float64 with an additive float mask
(ALiBi bias, -inf outside the window) and with one extra zero key / zero value whose additive
bias is the sink logit; closed forms for a zero query; the limits of the soft cap.
"""

import numpy as np
import pytest
import torch

from oracle import hadamard, int4_cache
from quantized_paged_kv_int4_gb300 import workloads


def _build(case, num_blocks=None):
    bt, nb = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=num_blocks, unused_fill=-1)
    _, _, slots = workloads.all_token_slots(bt, case.seq_lens)
    k, v = workloads.kv_vectors(case, slots.numel())
    Hk, D = case.Hk, case.D
    kc = np.zeros((nb, 16, Hk, D // 2), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nb, 16, Hk), np.uint32)
    vs = np.zeros_like(ks)
    sg = workloads.rht_signs(D).numpy()
    int4_cache.write_int4(workloads.to_numpy_f32(k), workloads.to_numpy_f32(v), slots.numpy(), sg, kc, vc, ks, vs)
    q = workloads.to_numpy_f32(workloads.query(case))
    return dict(q=q, kc=kc, vc=vc, ks=ks, vs=vs, bt=bt.numpy(), lens=np.array(case.seq_lens), signs=sg,
                Hq=case.Hq, Hk=Hk, D=D)


def _run(c, scale, **kw):
    return int4_cache.decode_int4(c["q"], c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["lens"],
                                  c["signs"], scale, **kw)


def _unrotate(x, signs, D):
    return (np.asarray(x, np.float64) @ hadamard.sylvester(D).T) * signs.astype(np.float64) / D


def _dequant_seq(c, b, pool, scales):
    L = int(c["lens"][b])
    rows = [int4_cache.dequant_int4(c[pool][c["bt"][b, n // 16], n % 16], c[scales][c["bt"][b, n // 16], n % 16])
            for n in range(L)]
    return np.stack([_unrotate(r, c["signs"], c["D"]) for r in rows])  # [L, Hk, D], original space


def _sdpa(c, scale, window=0, slopes=None, sinks=None):
    """Plain attention in the original space with the modifiers as an additive float mask."""
    Hq, Hk, D = c["Hq"], c["Hk"], c["D"]
    G = Hq // Hk
    q_rot = int4_cache.rotate_to_bf16(c["q"], c["signs"])
    out = np.zeros(c["q"].shape, np.float64)
    for b, L in enumerate(c["lens"]):
        if L == 0:
            continue
        Kt, Vt = _dequant_seq(c, b, "kc", "ks"), _dequant_seq(c, b, "vc", "vs")
        pos = np.arange(L, dtype=np.float64)
        bias = np.zeros((Hq, L))
        if slopes is not None:
            bias += np.asarray(slopes, np.float64)[:, None] * (pos - (L - 1))[None, :]
        if window > 0:
            bias[:, pos < L - window] = -np.inf
        K = np.repeat(Kt.transpose(1, 0, 2), G, axis=0)   # [Hq, L, D]
        V = np.repeat(Vt.transpose(1, 0, 2), G, axis=0)
        if sinks is not None:  # one more key: zero vector (score 0), bias = sink, zero value
            K = np.concatenate([K, np.zeros((Hq, 1, D))], axis=1)
            V = np.concatenate([V, np.zeros((Hq, 1, D))], axis=1)
            bias = np.concatenate([bias, np.asarray(sinks, np.float64)[:, None]], axis=1)
        Q = torch.from_numpy(_unrotate(q_rot[b], c["signs"], D))[:, None, :]   # [Hq, 1, D]
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, torch.from_numpy(K), torch.from_numpy(V), attn_mask=torch.from_numpy(bias)[:, None, :], scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out


def _case(seed=11):
    return workloads.DecodeCase("mods", 3, 8, 2, 64, [37, 100, 16], seed=seed)


def _slopes(Hq):
    return 2.0 ** (-8.0 * (np.arange(Hq) + 1) / Hq)   # the ALiBi geometric slopes


@pytest.mark.parametrize("window", [0, 1, 5, 16, 40, 1000])
def test_alibi_and_window_match_sdpa_with_additive_mask(window):
    c = _build(_case())
    scale = 1.0 / np.sqrt(64)
    sl = _slopes(c["Hq"])
    got = _run(c, scale, window=window, alibi_slopes=sl)
    assert np.max(np.abs(got - _sdpa(c, scale, window=window, slopes=sl))) < 1e-12
    if window:
        got = _run(c, scale, window=window)
        assert np.max(np.abs(got - _sdpa(c, scale, window=window))) < 1e-12


def test_sinks_match_sdpa_with_a_zero_value_key():
    c = _build(_case(12))
    scale = 1.0 / np.sqrt(64)
    sinks = np.linspace(-3.0, 4.0, c["Hq"])
    got = _run(c, scale, sinks=sinks)
    assert np.max(np.abs(got - _sdpa(c, scale, sinks=sinks))) < 1e-12
    sl = _slopes(c["Hq"])
    got = _run(c, scale, sinks=sinks, alibi_slopes=sl, window=21)
    assert np.max(np.abs(got - _sdpa(c, scale, window=21, slopes=sl, sinks=sinks))) < 1e-12


def test_softcap_limits():
    c = _build(_case(13))
    scale = 0.4
    plain = _run(c, scale)
    assert np.max(np.abs(_run(c, scale, softcap=1e7) - plain)) < 1e-9      # tanh(x) ~ x
    # a vanishing cap makes every kept score ~0: the output is the mean value of the kept keys
    got = _run(c, scale, softcap=1e-9, window=9)
    for b, L in enumerate(c["lens"]):
        Vt = _dequant_seq(c, b, "vc", "vs")[max(0, L - 9):]
        mean = np.repeat(Vt.mean(axis=0), c["Hq"] // c["Hk"], axis=0)
        assert np.max(np.abs(got[b] - mean)) < 1e-7
    # the cap comes before the ALiBi bias: with a vanishing cap only the bias weights the keys
    sl = _slopes(c["Hq"])
    got = _run(c, scale, softcap=1e-9, alibi_slopes=sl)
    G = c["Hq"] // c["Hk"]
    for b, L in enumerate(c["lens"]):
        Vt = _dequant_seq(c, b, "vc", "vs")
        for hq in range(c["Hq"]):
            w = np.exp(-sl[hq] * (L - 1 - np.arange(L)))
            assert np.max(np.abs(got[b, hq] - (w[:, None] * Vt[:, hq // G]).sum(axis=0) / w.sum())) < 1e-7
    # a moderate cap changes the result
    capped = _run(c, scale, softcap=0.5)
    assert np.max(np.abs(capped - plain)) > 1e-4


def test_zero_query_closed_forms():
    """q = 0: every score is 0, so the weights are the ALiBi factors r^(L-1-n) (r = e^-slope) and
    the sink adds e^sink to the denominator."""
    c = _build(_case(14))
    c["q"][:] = 0.0
    sl = _slopes(c["Hq"])
    sinks = np.linspace(-1.0, 2.0, c["Hq"])
    got = _run(c, 0.3, alibi_slopes=sl, sinks=sinks, window=30)
    G = c["Hq"] // c["Hk"]
    for b, L in enumerate(c["lens"]):
        Vt = _dequant_seq(c, b, "vc", "vs")
        lo = max(0, L - 30)
        for hq in range(c["Hq"]):
            w = np.exp(-sl[hq] * (L - 1 - np.arange(lo, L)))
            num = (w[:, None] * Vt[lo:, hq // G]).sum(axis=0)
            assert np.max(np.abs(got[b, hq] - num / (w.sum() + np.exp(sinks[hq])))) < 1e-12


def test_window_one_returns_the_last_value():
    c = _build(_case(15))
    got = _run(c, 0.2, window=1, softcap=3.0, alibi_slopes=_slopes(c["Hq"]))
    G = c["Hq"] // c["Hk"]
    for b, L in enumerate(c["lens"]):
        last = _dequant_seq(c, b, "vc", "vs")[L - 1]
        assert np.max(np.abs(got[b] - np.repeat(last, G, axis=0))) < 1e-12


@pytest.mark.parametrize("S", [1, 3, 7, 64])
def test_modifiers_split_merge_equals_single_pass(S):
    c = _build(_case(16))
    kw = dict(window=45, softcap=2.5, alibi_slopes=_slopes(c["Hq"]), sinks=np.linspace(-2, 2, c["Hq"]))
    assert np.max(np.abs(_run(c, 0.25, num_splits=S, **kw) - _run(c, 0.25, **kw))) < 1e-12
