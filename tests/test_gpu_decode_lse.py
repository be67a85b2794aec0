"""The merged log-sum-exp output of the decode calls (lse_out), against the float64 oracle.

triton_turboquant_decode.py, triton_turboquant_decode_attention returns lse_buf next to the
output so that a caller can merge the result with attention over other keys. The kernels keep
scores in base-2 units against a per-column reference; the merge writes (M + log2 den) ln 2.
Tolerance: 1e-4 absolute on the natural-log lse (fp32 sums of up to a few thousand terms)."""

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import Int4Case, TqCase, assert_close

pytestmark = pytest.mark.gpu

LENS = [1, 16, 17, 300, 0, 2049]


def _lse_close(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.array_equal(np.isinf(got), np.isinf(ref)), what
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin])
    assert err.max() < 1e-4, "%s: max lse err %.3e" % (what, err.max())


@pytest.mark.parametrize("S", [0, 3])
@pytest.mark.parametrize("with_sinks", [False, True])
def test_int4_lse_out(S, with_sinks):
    case = workloads.DecodeCase("lse", len(LENS), 32, 8, 128, LENS, seed=51, outlier_channels=4)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(LENS)) + 3)
    g = c.to_gpu()
    sinks = torch.randn((32,), generator=torch.Generator().manual_seed(3)) * 2.0 if with_sinks else None
    ref, ref_lse = c.oracle(return_lse=True, sinks=None if sinks is None else sinks.numpy())
    lse = torch.full((case.B, case.Hq), float("nan"), dtype=torch.float32, device="cuda")
    out = kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                              num_splits=S, sinks=None if sinks is None else sinks.cuda(), lse_out=lse)
    assert kvq.kvq_device_error() == (0, 0)
    assert_close(out.cpu().numpy(), ref, what="out S=%d sinks=%d" % (S, with_sinks))
    _lse_close(lse.cpu().numpy(), ref_lse, "lse S=%d sinks=%d" % (S, with_sinks))


def test_int4_lse_out_multi_token():
    Q = 2
    lens = [5, 40, 700]
    case = workloads.DecodeCase("lseq", len(lens), 8, 2, 64, lens, seed=52)
    c = Int4Case(case)
    c.q = workloads.bf16_normal((len(lens) * Q, 8, 64), 52, 1)
    g = c.to_gpu()
    ref, ref_lse = c.oracle(return_lse=True, q_len=Q)
    lse = torch.empty((len(lens) * Q, 8), dtype=torch.float32, device="cuda")
    out = kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                              q_len=Q, lse_out=lse)
    assert kvq.kvq_device_error() == (0, 0)
    assert_close(out.cpu().numpy(), ref, what="out Q=2")
    _lse_close(lse.cpu().numpy(), ref_lse, "lse Q=2")


@pytest.mark.parametrize("bits", [4, 3])
def test_tq_lse_out(bits):
    case = workloads.DecodeCase("tqlse", len(LENS), 32, 8, 128, LENS, seed=53 + bits)
    c = TqCase(case, bits, num_blocks=sum(workloads.pages_needed(LENS)) + 3)
    from oracle import turboquant
    ref, ref_lse = turboquant.decode_tq(c.q.numpy(), c.cache.numpy(), bits, c.bt.numpy(), np.asarray(LENS),
                                        c.scale, return_lse=True)
    for S in (0, 4):
        lse = torch.full((case.B, case.Hq), float("nan"), dtype=torch.float32, device="cuda")
        out = kvq.kvq_decode_tq(c.q.cuda(), c.cache.cuda(), bits, c.bt.cuda(), c.lens.cuda(), c.scale,
                                num_splits=S, lse_out=lse)
        assert kvq.kvq_device_error() == (0, 0)
        assert_close(out.cpu().numpy(), ref, what="tq out bits=%d S=%d" % (bits, S))
        _lse_close(lse.cpu().numpy(), ref_lse, "tq lse bits=%d S=%d" % (bits, S))
