"""kvq_decode_int4_noalloc: the decode for callers that cannot allocate device memory.

Such callers (for example a plug-in inside a serving process whose allocator already owns all of
HBM, or a C caller without the host framework's allocator) get the library's own device scratch
array instead of passing a workspace. These tests call that entry point through the C ABI and
check it against the float64 oracle and against the workspace entry point, on two calls in a row
(the second call finds the first call's leftovers in the shared array). The large balanced-split
case runs first, so the tiny fixed-split case that follows also starts on another layout's
leftovers. The file is named to be collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process, where its first call
is the one that looks up the array's device address.
"""

import ctypes

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import Int4Case, assert_close

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(g, scale, out, num_splits, dims):
    B, Hq, Hk, D, nb = dims
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return kvq.lib().kvq_decode_int4_noalloc(
        _ptr(g["q"]), _ptr(g["kc"]), _ptr(g["vc"]), _ptr(g["ks"]), _ptr(g["vs"]), _ptr(g["bt"]),
        g["bt"].shape[1], _ptr(g["lens"]), _ptr(g["signs"]), ctypes.c_float(scale), num_splits, _ptr(out),
        kvq.KVQ_F32, B, Hq, Hk, D, 16, nb, stream)


CASES = [  # the large balanced-split case first, then the tiny fixed-split one on its leftovers
    (workloads.DecodeCase("noalloc", 6, 32, 8, 128, [1024, 1500, 2049, 0, 3000, 1], seed=5,
                          outlier_channels=4), 0),
    (workloads.tiny_int4(), 4),
]


def test_noalloc_matches_the_oracle_twice_per_case():
    for case, num_splits in CASES:
        c = Int4Case(case)
        g = c.to_gpu()
        ref = c.oracle()
        ws = kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"],
                                 c.scale, num_splits=num_splits).cpu().numpy()
        dims = (case.B, case.Hq, case.Hk, case.D, c.nb)
        for _ in range(2):
            out = torch.full((case.B, case.Hq, case.D), float("nan"), dtype=torch.float32, device="cuda")
            assert _noalloc(g, c.scale, out, num_splits, dims) == kvq.KVQ_OK
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            assert_close(got, ref, what="noalloc vs oracle S=%d" % num_splits)
            assert_close(got, ws, what="noalloc vs workspace entry point S=%d" % num_splits)
        assert kvq.kvq_device_error() == (0, 0)


def test_noalloc_python_wrapper_and_its_checks():
    c = Int4Case(workloads.tiny_int4())
    g = c.to_gpu()
    out = torch.empty((c.case.B, c.case.Hq, c.case.D), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_int4_noalloc(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"],
                                c.scale, out, num_splits=4)
    assert_close(out.cpu().numpy(), c.oracle(), what="noalloc wrapper")
    with pytest.raises(ValueError):  # an output smaller than q is rejected before any launch
        kvq.kvq_decode_int4_noalloc(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"],
                                    c.scale, out[:1])
    with pytest.raises(TypeError):
        kvq.kvq_decode_int4_noalloc(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"],
                                    c.scale, out.to(torch.int32))


def test_noalloc_rejects_a_scratch_need_above_the_array():
    # 64 sequences x 64 query heads x 64 splits need ~135 MB of scratch: rejected before launch
    B, Hq, Hk, D, S = 64, 64, 8, 128, 64
    assert kvq.kvq_decode_workspace_bytes(B, Hq, Hk, D, S) > kvq.KVQ_NOALLOC_SCRATCH_BYTES
    lens = [32] * B
    case = workloads.DecodeCase("big", B, Hq, Hk, D, lens, seed=6)
    c = Int4Case(case, random_cache=True)
    g = c.to_gpu()
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda")
    assert _noalloc(g, c.scale, out, S, (B, Hq, Hk, D, c.nb)) == kvq.KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert np.all(out.cpu().numpy() == 0.0)
