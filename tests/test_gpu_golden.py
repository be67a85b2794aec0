"""The CUDA path against the stored oracle fixtures of tests/golden/ (see test_golden.py):
cache bytes, scale words and FP8 codes bit-exact; attention within the decode tolerance."""

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import kvq

from helpers import assert_close
from test_golden import _arr, _fixture

pytestmark = pytest.mark.gpu
F32 = np.float32


def _bf16(a_f32):
    return torch.from_numpy(a_f32).to(torch.bfloat16)  # exact: the values are bf16


def test_write_matches_fixture():
    f = _fixture("int4_write_tiny.json")
    T, Hk, D, nb = f["T"], f["Hk"], f["D"], f["num_blocks"]
    k = _bf16(_arr(f["key_bf16_as_f32"], F32, (T, Hk, D))).cuda()
    v = _bf16(_arr(f["value_bf16_as_f32"], F32, (T, Hk, D))).cuda()
    signs = torch.from_numpy(_arr(f["signs"], F32, (D,))).cuda()
    slots = torch.tensor(f["slot_mapping"], dtype=torch.int64, device="cuda")
    for name, sg in (("rotated", signs), ("plain", None)):
        kc = torch.zeros((nb, 16, Hk, D // 2), dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros((nb, 16, Hk), dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
        kvq.kvq_write_int4(k, v, kc, vc, ks, vs, slots, sg)
        torch.cuda.synchronize()
        exp = f[name]
        assert kc.cpu().numpy().tobytes().hex() == exp["k_cache"]
        assert vc.cpu().numpy().tobytes().hex() == exp["v_cache"]
        assert ks.cpu().numpy().tobytes().hex() == exp["k_scale"]
        assert vs.cpu().numpy().tobytes().hex() == exp["v_scale"]


@pytest.mark.parametrize("num_splits", [0, 2])
def test_decode_matches_fixture(num_splits):
    f = _fixture("int4_decode_tiny.json")
    B, Hq, Hk, D, nb = f["B"], f["Hq"], f["Hk"], f["D"], f["num_blocks"]
    t = lambda h, dt, shape: torch.from_numpy(_arr(f[h], dt, shape)).cuda()
    kc = t("k_cache", np.uint8, (nb, 16, Hk, D // 2))
    vc = t("v_cache", np.uint8, (nb, 16, Hk, D // 2))
    ks = torch.from_numpy(_arr(f["k_scale"], np.uint32, (nb, 16, Hk)).view(np.float32)).cuda()
    vs = torch.from_numpy(_arr(f["v_scale"], np.uint32, (nb, 16, Hk)).view(np.float32)).cuda()
    q = _bf16(_arr(f["q_bf16_as_f32"], F32, (B, Hq, D))).cuda()
    signs = t("signs", F32, (D,))
    bt = torch.tensor(f["block_table"], dtype=torch.int32, device="cuda")
    lens = torch.tensor(f["seq_lens"], dtype=torch.int32, device="cuda")
    for key, sg in (("out_rotated_f64", signs), ("out_plain_f64", None)):
        out = kvq.kvq_decode_int4(q, kc, vc, ks, vs, bt, lens, sg, f["softmax_scale"], num_splits=num_splits,
                                  out_dtype=torch.float32)
        assert_close(out.cpu().numpy(), _arr(f[key], np.float64, (B, Hq, D)), what=key)


def test_fwht_matches_fixture():
    f = _fixture("fwht128_fp8_tiny.json")
    x = _bf16(_arr(f["x_bf16_as_f32"], F32, (4, 128))).cuda()
    y, s = kvq.kvq_fwht128(x)
    torch.cuda.synchronize()
    assert y.view(torch.uint8).cpu().numpy().tobytes().hex() == f["y_e4m3"]
    assert s.cpu().numpy().tobytes().hex() == f["row_scale_f32"]


@pytest.mark.parametrize("bits", [4, 3])
def test_tq_matches_fixture(bits):
    f = _fixture("tq_decode_tiny.json")
    g = f["v%d" % bits]
    Hk, D, Hq = f["Hk"], f["D"], f["Hq"]
    cache = torch.from_numpy(_arr(g["kv_cache"], np.uint8, (1, 16, Hk, g["slot_bytes"]))).cuda()
    q = torch.from_numpy(_arr(g["q_f32"], F32, (1, Hq, D))).cuda()
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    lens = torch.tensor([g["seq_len"]], dtype=torch.int32, device="cuda")
    out = kvq.kvq_decode_tq(q, cache, bits, bt, lens, g["attn_scale"])
    assert_close(out.cpu().numpy(), _arr(g["out_f64"], np.float64, (1, Hq, D)), what="tq v%d" % bits)
