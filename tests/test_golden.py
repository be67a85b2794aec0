"""The oracle against tests/golden/: the constants the pages print (page_constants.txt) and the
stored oracle fixtures (written by tests/golden/make_golden.py), so a change to the oracle's
arithmetic shows up here. No GPU."""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats, fwht_fp8, hadamard, int4_cache, turboquant
from quantized_paged_kv_int4_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _constants():
    out = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, value, _ = line.split(" ", 2)
                out[name] = value
    return out


def _fixture(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _arr(hexstr, dtype, shape):
    return np.frombuffer(bytes.fromhex(hexstr), dtype=dtype).reshape(shape).copy()


def test_page_constants_in_the_oracle():
    c = _constants()
    # quantizer: scale = max((max - min) / 15, 1e-6), codes in [0, 15]
    _, w = int4_cache.quantize_int4(np.full((1, 64), 5.0, F32))
    floor = F32(float(c["int4_scale_floor"]))
    assert (w[0] & ~np.uint32(0xF)) == (floor.view(np.uint32) & ~np.uint32(0xF))
    q, w = int4_cache.quantize_int4(np.linspace(0.0, 30.0, 64, dtype=F32)[None])
    div = F32(float(c["int4_scale_divisor"]))
    assert (w[0] & ~np.uint32(0xF)) == ((F32(30.0) / div).view(np.uint32) & ~np.uint32(0xF))
    assert q.max() == int(c["int4_code_max"]) and q.min() == 0
    # FWHT-128: normalisation, absmax floor, e4m3 range
    assert hadamard.H128_SCALE_F32 == F32(float(c["fwht128_norm"]))
    y, s = fwht_fp8.fwht128_quant_fp8(np.zeros((1, 128), F32))
    assert s[0] == fwht_fp8.pow2_ceil(F32(float(c["fwht_absmax_floor"])) * (F32(1.0) / F32(float(c["fp8_e4m3_max"]))))
    x = np.zeros((1, 128), F32)
    x[0, 3] = F32(1e5)
    y, s = fwht_fp8.fwht128_quant_fp8(x)
    assert np.abs(formats.e4m3fn_to_f64(y)).max() <= float(c["fp8_e4m3_max"])
    # RHT signs: a CPU generator seeded with seed + round * stride, Bernoulli(1/2) mapped to +-1
    seed, stride = int(c["rht_seed"], 16), int(c["rht_round_stride"], 16)
    for rnd in (0, 1):
        g = torch.Generator().manual_seed(seed + rnd * stride)
        ref = 2.0 * torch.bernoulli(torch.full((128,), 0.5), generator=g) - 1.0
        assert torch.equal(workloads.rht_signs(128, rnd), ref)


def test_write_fixture():
    f = _fixture("int4_write_tiny.json")
    T, Hk, D, nb = f["T"], f["Hk"], f["D"], f["num_blocks"]
    k = _arr(f["key_bf16_as_f32"], F32, (T, Hk, D))
    v = _arr(f["value_bf16_as_f32"], F32, (T, Hk, D))
    signs = _arr(f["signs"], F32, (D,))
    for name, sg in (("rotated", signs), ("plain", None)):
        kc = np.zeros((nb, 16, Hk, D // 2), np.uint8)
        vc = np.zeros_like(kc)
        ks = np.zeros((nb, 16, Hk), np.uint32)
        vs = np.zeros_like(ks)
        int4_cache.write_int4(k, v, np.asarray(f["slot_mapping"]), sg, kc, vc, ks, vs)
        exp = f[name]
        assert kc.tobytes().hex() == exp["k_cache"] and vc.tobytes().hex() == exp["v_cache"]
        assert ks.tobytes().hex() == exp["k_scale"] and vs.tobytes().hex() == exp["v_scale"]


def test_decode_fixture():
    f = _fixture("int4_decode_tiny.json")
    B, Hq, Hk, D, nb = f["B"], f["Hq"], f["Hk"], f["D"], f["num_blocks"]
    kc = _arr(f["k_cache"], np.uint8, (nb, 16, Hk, D // 2))
    vc = _arr(f["v_cache"], np.uint8, (nb, 16, Hk, D // 2))
    ks = _arr(f["k_scale"], np.uint32, (nb, 16, Hk))
    vs = _arr(f["v_scale"], np.uint32, (nb, 16, Hk))
    q = _arr(f["q_bf16_as_f32"], F32, (B, Hq, D))
    signs = _arr(f["signs"], F32, (D,))
    bt, lens = np.asarray(f["block_table"], np.int32), np.asarray(f["seq_lens"])
    for key, sg in (("out_rotated_f64", signs), ("out_plain_f64", None)):
        got = int4_cache.decode_int4(q, kc, vc, ks, vs, bt, lens, sg, f["softmax_scale"])
        np.testing.assert_allclose(got, _arr(f[key], np.float64, (B, Hq, D)), rtol=1e-12, atol=1e-14)


def test_fwht_fixture():
    f = _fixture("fwht128_fp8_tiny.json")
    x = _arr(f["x_bf16_as_f32"], F32, (4, 128))
    y, s = fwht_fp8.fwht128_quant_fp8(x)
    assert y.tobytes().hex() == f["y_e4m3"] and s.tobytes().hex() == f["row_scale_f32"]


@pytest.mark.parametrize("bits", [4, 3])
def test_tq_fixture(bits):
    f = _fixture("tq_decode_tiny.json")
    g = f["v%d" % bits]
    Hk, D, Hq = f["Hk"], f["D"], f["Hq"]
    cache = _arr(g["kv_cache"], np.uint8, (1, 16, Hk, g["slot_bytes"]))
    q = _arr(g["q_f32"], F32, (1, Hq, D))
    got = turboquant.decode_tq(q, cache, bits, np.array([[0]], np.int32), np.array([g["seq_len"]]), g["attn_scale"])
    np.testing.assert_allclose(got, _arr(g["out_f64"], np.float64, (1, Hq, D)), rtol=1e-12, atol=1e-14)
    assert math.isclose(g["attn_scale"], 1.0 / math.sqrt(D))
