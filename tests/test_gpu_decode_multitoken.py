"""Multi-token INT4 decode on the GPU against the float64 oracle: q_len query tokens per sequence
(the speculative-verify case) and ragged per-sequence counts (query_start_loc, chunked prefill),
causal, with the score modifiers per query token. Tolerance: 2e-3 + 1e-2 |oracle| elementwise."""

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import Int4Case, assert_close

pytestmark = pytest.mark.gpu


def _queries(B, Q, Hq, D, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((B * Q, Hq, D), generator=g).to(torch.bfloat16)


def _run(c, q, Q, num_splits=0, **mods):
    g = c.to_gpu()
    out = kvq.kvq_decode_int4(q.cuda(), g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                              num_splits=num_splits, out_dtype=torch.float32, q_len=Q, **mods)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0, (st, flags)
    return out.cpu().numpy()


def _oracle(c, q, Q, **mods):
    from oracle import int4_cache
    m = {("window" if k == "sliding_window" else k): (v.numpy() if isinstance(v, torch.Tensor) else v)
         for k, v in mods.items()}
    return int4_cache.decode_int4(workloads.to_numpy_f32(q), c.kc, c.vc, c.ks, c.vs, c.bt.numpy(),
                                  np.asarray(c.case.seq_lens), c.signs.numpy(), c.scale, q_len=Q, **m)


@pytest.mark.parametrize("Hk,G,Q,D", [(8, 4, 2, 128), (2, 2, 4, 64), (1, 1, 8, 128), (4, 2, 3, 128), (16, 1, 5, 64)])
def test_layouts_and_causal_edges(Hk, G, Q, D):
    """Lengths below, at and just past Q and around page boundaries; balanced and fixed splits."""
    lens = [1, Q, Q + 1, 16, 17, 15 + Q, 200, 0, 63]
    case = workloads.DecodeCase("mt", len(lens), Hk * G, Hk, D, lens, seed=Hk * 13 + G * 3 + Q)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(lens)) + 4)
    q = _queries(len(lens), Q, Hk * G, D, seed=Q)
    ref = _oracle(c, q, Q)
    for S in (0, 3):
        got = _run(c, q, Q, num_splits=S)
        assert_close(got, ref, what="Hk=%d G=%d Q=%d D=%d S=%d" % (Hk, G, Q, D, S))
        assert np.all(got[7 * Q:8 * Q] == 0.0)


def test_with_softcap_and_sinks():
    lens = [5, 100, 33]
    case = workloads.DecodeCase("mtm", 3, 8, 4, 128, lens, seed=5)
    c = Int4Case(case)
    q = _queries(3, 4, 8, 128, seed=6)
    sinks = torch.linspace(-2.0, 3.0, 8)
    mods = dict(softcap=4.0, sinks=sinks)
    got = _run(c, q, 4, softcap=4.0, sinks=sinks.cuda())
    assert_close(got, _oracle(c, q, 4, **mods), what="Q=4 cap + sinks")


def test_q_len_one_equals_the_single_token_call():
    case = workloads.DecodeCase("mt1", 3, 8, 2, 64, [40, 300, 7], seed=7)
    c = Int4Case(case)
    g = c.to_gpu()
    a = kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                            out_dtype=torch.float32).cpu().numpy()
    b = kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                            out_dtype=torch.float32, q_len=1).cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("Q", [4, 9])
def test_more_query_columns_than_the_mma_has(Q):
    """G * Q = 16 and 36 columns: the tokens are served in blocks of 8 / G = 2 (BLOCK_Q tiling)."""
    lens = [40, 70, Q, 300]
    case = workloads.DecodeCase("mtq", len(lens), 32, 8, 128, lens, seed=8 + Q)
    c = Int4Case(case)
    q = _queries(len(lens), Q, 32, 128, seed=9)
    ref = _oracle(c, q, Q)
    for S in (0, 2):
        assert_close(_run(c, q, Q, num_splits=S), ref, what="G*Q=%d S=%d" % (4 * Q, S))


@pytest.mark.parametrize("S", [0, 3])
def test_window_and_alibi_per_query_token(S):
    """Each query token's window and ALiBi bias are taken at its own position."""
    lens = [5, 100, 33, 64]
    case = workloads.DecodeCase("mtw", len(lens), 16, 4, 128, lens, seed=12)
    c = Int4Case(case)
    q = _queries(len(lens), 3, 16, 128, seed=13)
    slopes = 2.0 ** (-8.0 * (torch.arange(16, dtype=torch.float32) + 1) / 16)
    for mods in (dict(sliding_window=20), dict(alibi_slopes=slopes), dict(sliding_window=7, alibi_slopes=slopes,
                                                                          softcap=5.0)):
        m = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in mods.items()}
        assert_close(_run(c, q, 3, num_splits=S, **m), _oracle(c, q, 3, **mods), what="%s S=%d" % (list(mods), S))


def _ragged(counts, lens, Hq, Hk, D, seed, num_splits=0, **mods):
    case = workloads.DecodeCase("rag", len(lens), Hq, Hk, D, lens, seed=seed, outlier_channels=4)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(lens)) + 3)
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    q = _queries(1, int(qsl[-1]), Hq, D, seed=seed + 1)
    g = c.to_gpu()
    m = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in mods.items()}
    out = kvq.kvq_decode_int4(q.cuda(), g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                              num_splits=num_splits, out_dtype=torch.float32, query_start_loc=qsl.cuda(), **m)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0, (st, flags)
    from oracle import int4_cache
    om = {("window" if k == "sliding_window" else k): (v.numpy() if isinstance(v, torch.Tensor) else v)
          for k, v in mods.items()}
    ref = int4_cache.decode_int4(workloads.to_numpy_f32(q), c.kc, c.vc, c.ks, c.vs, c.bt.numpy(),
                                 np.asarray(lens), c.signs.numpy(), c.scale, query_start_loc=qsl.numpy(), **om)
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("Hk,G,D", [(8, 4, 128), (2, 8, 64), (4, 1, 128)])
@pytest.mark.parametrize("S", [0, 2])
def test_ragged_query_counts(Hk, G, D, S):
    """Per-sequence query counts 0, 1, 2, 7, 8/G + 1 and 20 (chunked-prefill-like) in one batch, with
    lengths around page edges; the varlen query_start_loc layout."""
    counts = [0, 1, 2, 7, 8 // G + 1, 20, 3]
    lens = [10, 1, 17, 40, 33, 300, 3]
    got, ref = _ragged(counts, lens, Hk * G, Hk, D, seed=20 + G, num_splits=S)
    assert_close(got, ref, what="ragged Hk=%d G=%d S=%d" % (Hk, G, S))


def test_ragged_with_every_modifier_and_lse():
    counts = [3, 0, 5, 1, 12]
    lens = [9, 40, 17, 3, 700]
    Hq = 16
    slopes = 2.0 ** (-8.0 * (torch.arange(Hq, dtype=torch.float32) + 1) / Hq)
    sinks = torch.linspace(-1.0, 2.0, Hq)
    got, ref = _ragged(counts, lens, Hq, 4, 128, seed=31, sliding_window=6, alibi_slopes=slopes, softcap=8.0,
                       sinks=sinks)
    assert_close(got, ref, what="ragged + all modifiers")


def test_llama8b_shaped_two_token_verify_sampled():
    """B=32, Hq=32, Hk=8, D=128, L ~ U[1024, 8192], two query tokens per sequence (G * Q = 8)."""
    case = workloads.llama8b_int4()
    c = Int4Case(case, random_cache=True)
    q = _queries(case.B, 2, 32, 128, seed=10)
    got = _run(c, q, 2)
    from oracle import int4_cache
    idx = [0, 13, 31]
    ref = int4_cache.decode_int4(workloads.to_numpy_f32(q), c.kc, c.vc, c.ks, c.vs, c.bt.numpy(),
                                 np.asarray(case.seq_lens), c.signs.numpy(), c.scale, q_len=2, batch_index=idx)
    rows = [b * 2 + i for b in idx for i in range(2)]
    assert_close(got[rows], ref[rows], what="llama8b Q=2")
