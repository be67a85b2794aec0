"""kvq_decode_int4 with score modifiers (kvq_decode_int4_mods: sliding window, soft cap, ALiBi,
attention sinks) on the GPU against the float64 oracle on the same cache.

Tolerance as the plain decode: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise."""

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import Int4Case, assert_close, run_int4

pytestmark = pytest.mark.gpu

LENS = [1, 15, 16, 17, 200, 513, 0, 33, 1000]


def _slopes(Hq):
    return (2.0 ** (-8.0 * (np.arange(Hq) + 1) / Hq)).astype(np.float32)


def _sinks(Hq, seed):
    return (np.random.default_rng(seed).standard_normal(Hq) * 2.0).astype(np.float32)


def _both(c, mods_np, num_splits, what, batch_index=None):
    """Run GPU and oracle with the same modifiers (numpy arrays -> device tensors for the GPU)."""
    g = c.to_gpu()
    mods_gpu = {k: (torch.from_numpy(v).cuda() if isinstance(v, np.ndarray) else v) for k, v in mods_np.items()}
    got = run_int4(kvq, g, c.scale, num_splits=num_splits, **mods_gpu).cpu().numpy()
    orc = {"sliding_window": "window", "softcap": "softcap", "sinks": "sinks", "alibi_slopes": "alibi_slopes"}
    ref = c.oracle(batch_index=batch_index, **{orc[k]: v for k, v in mods_np.items()})
    if batch_index is not None:
        got, ref = got[batch_index], ref[batch_index]
    assert_close(got, ref, what=what)
    return got


@pytest.mark.parametrize("num_splits", [0, 5])
@pytest.mark.parametrize("mod", ["window", "softcap", "alibi", "sinks", "all"])
def test_each_modifier(mod, num_splits):
    case = workloads.DecodeCase("mods", len(LENS), 32, 8, 128, LENS, seed=21, outlier_channels=4)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(LENS)) + 5)
    Hq = case.Hq
    mods = {"window": dict(sliding_window=100), "softcap": dict(softcap=2.0),
            "alibi": dict(alibi_slopes=_slopes(Hq)), "sinks": dict(sinks=_sinks(Hq, 1)),
            "all": dict(sliding_window=333, softcap=5.0, alibi_slopes=_slopes(Hq), sinks=_sinks(Hq, 2))}[mod]
    got = _both(c, mods, num_splits, "%s S=%d" % (mod, num_splits))
    assert np.all(got[6] == 0.0)  # empty sequence


@pytest.mark.parametrize("window", [1, 15, 16, 17, 31, 200, 10 ** 6])
def test_window_edges(window):
    """Windows that start inside, at and just past a page boundary, and one longer than every
    sequence; balanced and fixed splits."""
    case = workloads.DecodeCase("win", len(LENS), 8, 2, 64, LENS, seed=22)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(LENS)) + 3)
    for S in (0, 3, 64):
        _both(c, dict(sliding_window=window), S, "window=%d S=%d" % (window, S))


@pytest.mark.parametrize("Hk,G,D", [(1, 8, 128), (2, 3, 64), (4, 2, 128), (16, 2, 64), (16, 5, 128)])
def test_all_modifiers_head_layouts(Hk, G, D):
    lens = [5, 16, 100, 257, 0, 64]
    case = workloads.DecodeCase("mhl", len(lens), Hk * G, Hk, D, lens, seed=Hk * 7 + G)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(lens)) + 4)
    Hq = case.Hq
    mods = dict(sliding_window=70, softcap=3.0, alibi_slopes=_slopes(Hq), sinks=_sinks(Hq, Hk + G))
    for S in (0, 2):
        _both(c, mods, S, "Hk=%d G=%d D=%d S=%d" % (Hk, G, D, S))


def test_peaky_scores_with_cap_and_bias():
    """A 30x softmax scale: the cap bounds the scores, the bias reshapes them; the running max moves."""
    case = workloads.DecodeCase("pk", 4, 32, 8, 128, [1000, 64, 4000, 17], seed=23, outlier_channels=4)
    c = Int4Case(case, scale_mult=30.0)
    _both(c, dict(softcap=10.0, alibi_slopes=_slopes(32)), 0, "peaky capped")
    _both(c, dict(alibi_slopes=_slopes(32) * 8.0), 0, "peaky steep bias")


def test_llama8b_full_size_with_modifiers_sampled():
    """The Llama-3-8B-shaped step (B=32, L ~ U[1024, 8192]) with a 4096-key window, cap 30,
    ALiBi and sinks: the benchmark's launch, oracle on sampled sequences."""
    case = workloads.llama8b_int4()
    c = Int4Case(case, random_cache=True)
    mods = dict(sliding_window=4096, softcap=30.0, alibi_slopes=_slopes(32), sinks=_sinks(32, 3))
    _both(c, mods, 0, "llama8b mods", batch_index=[0, 13, 31])


def test_modifiers_off_equal_the_plain_call():
    """Zero window / cap and no arrays take the plain entry point: identical bytes."""
    case = workloads.DecodeCase("off", 3, 8, 2, 64, [40, 300, 7], seed=24)
    c = Int4Case(case)
    g = c.to_gpu()
    a = run_int4(kvq, g, c.scale).cpu().numpy()
    b = run_int4(kvq, g, c.scale, sliding_window=0, softcap=0.0).cpu().numpy()
    assert np.array_equal(a, b)
    # a window as long as every sequence selects the same keys through the window path
    w = run_int4(kvq, g, c.scale, sliding_window=10 ** 6).cpu().numpy()
    assert_close(w, a, atol=1e-5, rtol=1e-5, what="window >= L")
