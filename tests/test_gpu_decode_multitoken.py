"""Multi-token INT4 decode (q_len query tokens per sequence, causal; the speculative-verify case)
on the GPU against the float64 oracle. Tolerance: 2e-3 + 1e-2 |oracle| elementwise."""

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


def test_unsupported_combinations_are_refused():
    case = workloads.DecodeCase("mtu", 2, 32, 8, 128, [40, 70], seed=8)
    c = Int4Case(case)
    q = _queries(2, 4, 32, 128, seed=9)   # G * Q = 16 columns
    with pytest.raises(kvq.KvqError):
        _run(c, q, 4)
    q = _queries(2, 2, 32, 128, seed=9)
    with pytest.raises(kvq.KvqError):
        _run(c, q, 2, sliding_window=16)


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
