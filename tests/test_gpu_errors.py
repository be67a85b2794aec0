"""Device-side index checks: bad block ids, slots beyond the pool and over-long sequences are
skipped and reported through kvq_device_error, and the context stays usable. Every access the
kernels make for these inputs stays inside the caller's buffers (the checks run before the
address is formed), so nothing here can fault."""

import math

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import Int4Case, run_int4

pytestmark = pytest.mark.gpu


def test_bad_block_id_is_flagged():
    c = Int4Case(workloads.tiny_int4())
    g = c.to_gpu()
    g["bt"][0, 1] = -7
    g["bt"][1, 2] = c.nb + 3
    kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale)
    st, flags = kvq.kvq_device_error()
    assert st == kvq.KVQ_ERR_OUT_OF_RANGE and flags & 1
    assert kvq.kvq_device_error() == (0, 0)  # cleared; later calls still work
    g["bt"] = c.bt.cuda()
    run_int4(kvq, g, c.scale)


def test_long_sequence_is_clamped_and_flagged():
    c = Int4Case(workloads.tiny_int4())
    g = c.to_gpu()
    g["lens"][1] = 16 * g["bt"].shape[1] + 50
    kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale)
    st, flags = kvq.kvq_device_error()
    assert st == kvq.KVQ_ERR_OUT_OF_RANGE and flags & 2


def test_slot_beyond_pool_is_flagged_and_skipped():
    k, v, slots, nb = workloads.write_case(T=40, Hk=2, D=64, hole_frac=0.0)
    slots[3] = nb * 16 + 5
    kc = torch.zeros((nb, 16, 2, 32), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((nb, 16, 2), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    kvq.kvq_write_int4(k.cuda(), v.cuda(), kc, vc, ks, vs, slots.cuda(), workloads.rht_signs(64).cuda())
    st, flags = kvq.kvq_device_error()
    assert st == kvq.KVQ_ERR_OUT_OF_RANGE and flags == 4
    written = (ks.view(torch.int32) != 0).sum().item()
    assert written == 39 * 2


def test_invalid_arguments_raise():
    q = torch.zeros((2, 4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        kvq.kvq_decode_int4(q, None, None, None, None, None, None, None, 0.1)
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        kvq.kvq_fwht128(x)
    c = Int4Case(workloads.tiny_int4())
    g = c.to_gpu()
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                            workspace=torch.empty((16,), dtype=torch.uint8, device="cuda"))
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE


def test_a_wait_that_runs_out_is_reported_and_the_gpu_stays_usable():
    """The bounded-wait path: the next call withholds one ring stage's page copies in its first CTA
    (kvq_debug_set_wait), so that CTA's waits on it run out after 5 ms; the call still returns,
    flag 8 is raised, and the following call on the same context is exact again."""
    lens = [1200, 700, 2000]
    case = workloads.DecodeCase("timeout", len(lens), 32, 8, 128, lens, seed=61, outlier_channels=4)
    c = Int4Case(case)
    g = c.to_gpu()
    try:
        kvq.kvq_debug_set_wait(5_000_000, 2)  # the first CTA (sequence 0, split 0) has 38 pages = 38 stages
        kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale,
                            num_splits=2)
        st, flags = kvq.kvq_device_error()
        assert st == kvq.KVQ_ERR_OUT_OF_RANGE and flags == 8, (st, flags)
    finally:
        kvq.kvq_debug_set_wait(0, -1)
    from helpers import assert_close
    for S in (2, 0):
        assert_close(run_int4(kvq, g, c.scale, num_splits=S).cpu().numpy(), c.oracle(), what="after the timeout")


@pytest.mark.parametrize("kind", ["fp8", "mse"])
def test_turboquant_wait_that_runs_out_is_reported(kind):
    """The TurboQuant kernels' bounded waits: the next call withholds ring tile 2 of the first CTA's
    first warp (its page copy is never issued), the wait on it runs out after 5 ms, flag 8 is
    raised, and the following call on the same context is exact again."""
    from helpers import MseCase, TqCase, assert_close
    lens = [1200, 700, 2000]
    case = workloads.DecodeCase("tqtimeout", len(lens), 32, 8, 128, lens, seed=62)
    if kind == "fp8":
        c = TqCase(case, 4)

        def call():
            return kvq.kvq_decode_tq(c.q.cuda(), c.cache.cuda(), c.bits, c.bt.cuda(), c.lens.cuda(), c.scale,
                                     num_splits=2)

        def ref():
            return c.oracle()
    else:
        c = MseCase(case, 3, 4)

        def call():
            return kvq.kvq_decode_tq_mse(c.q.cuda(), c.Pi.cuda(), c.cb.cuda(), c.cache.cuda(), c.kb, c.kps, c.vb,
                                         c.bt.cuda(), c.lens.cuda(), c.scale, num_splits=2)

        def ref():
            return c.oracle(False)
    try:
        kvq.kvq_debug_set_wait(5_000_000, 2)  # split 0 of sequence 0: 38 pages, one ring tile each per warp
        call()
        st, flags = kvq.kvq_device_error()
        assert st == kvq.KVQ_ERR_OUT_OF_RANGE and flags == 8, (st, flags)
    finally:
        kvq.kvq_debug_set_wait(0, -1)
    got = call()
    assert kvq.kvq_device_error() == (0, 0)
    assert_close(got.cpu().numpy(), ref(), what="%s after the timeout" % kind)
