"""Dynamic range of the decode kernels' fp16 tensor-core operands, against the float64 oracle.

The pages keep the value-weighted probabilities in fp32 (int4_per_token_head.py, _attn_packed:
P_v = P * v_token_head_scales in fp32, fed to tl.dot; triton_turboquant_decode.py,
_tq_decode_stage1 accumulates p * (idx * scale + zero) in fp32) and the query in fp32/bf16.
The kernels feed fp16 operands, so they must shift queries and weights into the fp16 range
(per-piece powers of two and the per-column softmax reference): these cases put value scales
from 2^-20 to ~1e7, mixed within one page, and queries from 1e-6 to 1e4 through each kernel.
The data are scaled copies of the usual seeded inputs; since the output scales with the values,
the tolerance 2e-3 + 1e-2 |oracle| is applied to (output / value magnitude).
"""

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import Int4Case, MseCase, TqCase, assert_close, assert_close_scaled, run_int4

pytestmark = pytest.mark.gpu

LENS = [1, 17, 300, 1200, 0, 64]


def _int4_case(seed, kv_transform=None, q_mult=1.0, G=4, Hk=8, D=128):
    case = workloads.DecodeCase("range", len(LENS), Hk * G, Hk, D, LENS, seed=seed, outlier_channels=4)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(LENS)) + 3, kv_transform=kv_transform)
    if q_mult != 1.0:
        c.q = (c.q.float() * q_mult).to(torch.bfloat16)
    return c


def _int4_all_splits(c, unit, what):
    g = c.to_gpu()
    ref = c.oracle()
    assert np.all(np.isfinite(ref))
    for S in (0, 3):
        got = run_int4(kvq, g, c.scale, num_splits=S).cpu().numpy()
        assert np.all(np.isfinite(got)), what
        assert_close_scaled(got, ref, unit, what="%s S=%d" % (what, S))


@pytest.mark.parametrize("F", [1e5, 1e7])
def test_int4_large_value_range(F):
    """V rows of magnitude ~F (per-token scale words ~0.4 F): P_v = p * scale_v far beyond fp16."""
    c = _int4_case(31, kv_transform=lambda k, v: (k, (v.float() * F).to(torch.bfloat16)))
    _int4_all_splits(c, F, "V x %g" % F)


def test_int4_mixed_value_scales_in_one_page():
    """Per-token value magnitudes 10^U(-3, 6) side by side in every page."""
    def tr(k, v):
        g = torch.Generator().manual_seed(7)
        e = torch.rand((v.shape[0], v.shape[1], 1), generator=g) * 9.0 - 3.0
        return k, (v.float() * torch.pow(10.0, e)).to(torch.bfloat16)
    c = _int4_case(32, kv_transform=tr)
    _int4_all_splits(c, 1e6, "mixed V scales")


def test_int4_small_value_range():
    """V of magnitude ~1e-6 (scale words a few times the writer's 1e-6 floor): p * scale_v would
    sit deep in fp16's subnormal range."""
    c = _int4_case(33, kv_transform=lambda k, v: (k, (v.float() * 1e-6).to(torch.bfloat16)))
    _int4_all_splits(c, 1e-6, "V x 1e-6")


@pytest.mark.parametrize("qm", [1e4, 1e-6])
@pytest.mark.parametrize("G,Hk,D", [(4, 8, 128), (8, 2, 64)])
def test_int4_query_range(qm, G, Hk, D):
    """q x 1e4 (|H(q d1)| up to ~1e6, beyond fp16) and q x 1e-6 (deep in fp16's subnormal range)."""
    c = _int4_case(34 + G, q_mult=qm, G=G, Hk=Hk, D=D)
    _int4_all_splits(c, 1.0, "q x %g G=%d" % (qm, G))


def test_int4_large_key_range():
    """K x 1e4 with V x 1e5: a peaky softmax whose weights also carry huge value scales."""
    c = _int4_case(36, kv_transform=lambda k, v: ((k.float() * 1e4).to(torch.bfloat16),
                                                   (v.float() * 1e5).to(torch.bfloat16)))
    _int4_all_splits(c, 1e5, "K x 1e4, V x 1e5")


def test_int4_absurd_query_raises_the_range_flag():
    """|q| ~ 1e35 (bf16) is beyond the supported query range (~2^100): the call reports flag 16
    instead of returning a silently wrong answer."""
    c = _int4_case(37, q_mult=1e35)
    g = c.to_gpu()
    kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale)
    st, flags = kvq.kvq_device_error()
    assert st == kvq.KVQ_ERR_OUT_OF_RANGE and flags & 16, (st, flags)
    # the context stays usable: the next normal call is exact again
    c2 = _int4_case(38)
    assert_close(run_int4(kvq, c2.to_gpu(), c2.scale).cpu().numpy(), c2.oracle(), what="after flag")


# ---------------------------------------------------------------------------------------------
# TurboQuant layouts: fp16 value scale / zero words patched into the seeded slots
# ---------------------------------------------------------------------------------------------
def _patch_tq_scales(cache, D, bits, scale_of, zero=0.0, seed=5):
    """Overwrite every slot's fp16 value scale with scale_of(shape) and its zero with `zero`."""
    vdb = -(-D * bits // 8)
    shape = cache.shape[:3]
    sc = torch.as_tensor(scale_of(shape, seed), dtype=torch.float32).to(torch.float16)
    zr = torch.full(shape, zero, dtype=torch.float16)
    cache[..., D + vdb:D + vdb + 2] = sc.view(torch.uint8).view(*shape, 2)
    cache[..., D + vdb + 2:D + vdb + 4] = zr.view(torch.uint8).view(*shape, 2)
    return cache


def _tq(c, S):
    out = kvq.kvq_decode_tq(c.q.cuda(), c.cache.cuda(), c.bits, c.bt.cuda(), c.lens.cuda(), c.scale,
                            num_splits=S)
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0, (st, flags)
    return out.cpu().numpy()


def _uniform_log(lo, hi):
    def f(shape, seed):
        g = torch.Generator().manual_seed(seed)
        return torch.pow(2.0, torch.rand(shape, generator=g) * (hi - lo) + lo)
    return f


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("lo,hi,unit", [(-20.0, -15.0, 2.0 ** -15 * 8), (10.0, 15.9, 2.0 ** 15.9 * 8),
                                        (-20.0, 15.9, 2.0 ** 15.9 * 8)])
def test_tq_value_scale_range(bits, lo, hi, unit):
    """fp16 value scales 2^lo .. 2^hi (subnormal to near fp16's maximum; mixed within pages)."""
    case = workloads.DecodeCase("tqr", len(LENS), 32, 8, 128, LENS, seed=40 + bits)
    c = TqCase(case, bits, num_blocks=sum(workloads.pages_needed(LENS)) + 3)
    c.cache = _patch_tq_scales(c.cache, 128, bits, _uniform_log(lo, hi), zero=0.0)
    ref = c.oracle()
    for S in (0, 3):
        assert_close_scaled(_tq(c, S), ref, unit, what="tq bits=%d scales 2^%g..2^%g S=%d" % (bits, lo, hi, S))


@pytest.mark.parametrize("qm", [1e4, 1e-6])
def test_tq_query_range(qm):
    """fp32 q x 1e4 (hi parts beyond fp16) and x 1e-6 (below fp16's normal range)."""
    case = workloads.DecodeCase("tqq", len(LENS), 32, 8, 128, LENS, seed=43)
    c = TqCase(case, 4, num_blocks=sum(workloads.pages_needed(LENS)) + 3)
    c.q = c.q * qm
    ref = c.oracle()
    for S in (0, 3):
        assert_close(_tq(c, S), ref, what="tq q x %g S=%d" % (qm, S))


@pytest.mark.parametrize("cm,qm", [(1e5, 1.0), (1e-5, 1.0), (1.0, 1e4), (1.0, 1e-6)])
def test_tq_mse_centroid_and_query_range(cm, qm):
    """MSE keys: centroids x 1e5 / 1e-5 and q x 1e4 / 1e-6 through the fp16 hi + lo operands."""
    case = workloads.DecodeCase("mser", len(LENS), 32, 8, 128, LENS, seed=44)
    c = MseCase(case, 3, 4, num_blocks=sum(workloads.pages_needed(LENS)) + 3)
    c.cb = c.cb * cm
    c.q = c.q * qm
    for corr in (False, True):
        assert_close(c.gpu(corr), c.oracle(corr), what="mse c x %g q x %g corr=%d" % (cm, qm, corr))


def test_tq_mse_value_scale_range():
    """MSE keys with fp16 value scales from 2^-20 to 2^15.9 mixed within pages."""
    case = workloads.DecodeCase("msev", len(LENS), 32, 8, 128, LENS, seed=45)
    c = MseCase(case, 3, 4, num_blocks=sum(workloads.pages_needed(LENS)) + 3)
    mse, kps, sb = workloads.turboquant_mse_layout(128, 3, 4)
    vdb = 64
    shape = c.cache.shape[:3]
    sc = _uniform_log(-20.0, 15.9)(shape, 9).to(torch.float16)
    c.cache[..., kps + vdb:kps + vdb + 2] = sc.view(torch.uint8).view(*shape, 2)
    unit = 2.0 ** 15.9 * 16
    for corr in (False, True):
        assert_close_scaled(c.gpu(corr), c.oracle(corr), unit, what="mse value scales corr=%d" % corr)
