"""Writes the oracle fixtures of tests/golden/ (run from the repository root:
`python tests/golden/make_golden.py`). Calls only oracle/ and numpy; inputs come from a seeded
numpy generator and are stored with the outputs, so a fixture is self-contained text.

Fixtures:
  int4_write_tiny.json   reshape_and_cache_int4 of 3 tokens x 2 kv heads x D=64, one slot
                         skipped, with and without the rotation: packed bytes and scale words;
  int4_decode_tiny.json  paged decode over a 3-page pool (B=2, Hq=4, Hk=2, D=64, lens 3 and 20);
  fwht128_fp8_tiny.json  the fused FWHT-128 + pow2 FP8 quantizer on 4 rows;
  tq_decode_tiny.json    TurboQuant decode (FP8 keys, 4-bit and 3-bit values) on one page.
"""

import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import formats, fwht_fp8, int4_cache, turboquant  # noqa: E402

F32 = np.float32


def bf16_inputs(rng, shape, scale=1.0):
    return formats.bf16_round(rng.standard_normal(shape).astype(F32) * F32(scale))


def hexs(a):
    return np.ascontiguousarray(a).tobytes().hex()


def write_fixture(rng):
    T, Hk, D, nb = 3, 2, 64, 2
    k = bf16_inputs(rng, (T, Hk, D))
    v = bf16_inputs(rng, (T, Hk, D), 3.0)
    k[1, 0, 5] = F32(40.0)  # an outlier channel
    signs = np.where(rng.random(D) < 0.5, F32(-1.0), F32(1.0)).astype(F32)
    slots = np.array([5, -1, 18], dtype=np.int64)
    out = {}
    for name, sg in (("rotated", signs), ("plain", None)):
        kc = np.zeros((nb, 16, Hk, D // 2), np.uint8)
        vc = np.zeros_like(kc)
        ks = np.zeros((nb, 16, Hk), np.uint32)
        vs = np.zeros_like(ks)
        int4_cache.write_int4(k, v, slots, sg, kc, vc, ks, vs)
        out[name] = {"k_cache": hexs(kc), "v_cache": hexs(vc), "k_scale": hexs(ks), "v_scale": hexs(vs)}
    return {"T": T, "Hk": Hk, "D": D, "num_blocks": nb, "block_size": 16,
            "key_bf16_as_f32": hexs(k), "value_bf16_as_f32": hexs(v), "signs": hexs(signs),
            "slot_mapping": slots.tolist(), **out}


def decode_fixture(rng):
    B, Hq, Hk, D, nb = 2, 4, 2, 64, 3
    lens = np.array([3, 20], dtype=np.int64)
    bt = np.array([[2, 0], [1, 2]], dtype=np.int32)  # sequence 1 pages: 1 then 2 (rows 0..3)
    kc = rng.integers(0, 256, size=(nb, 16, Hk, D // 2), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(nb, 16, Hk, D // 2), dtype=np.uint8)
    scale = (rng.random((nb, 16, Hk)) * 0.2 + 0.05).astype(F32)
    zp = rng.integers(0, 16, size=(nb, 16, Hk), dtype=np.uint32)
    ks = (scale.view(np.uint32) & np.uint32(0xFFFFFFF0)) | zp
    scale = (rng.random((nb, 16, Hk)) * 0.3 + 0.05).astype(F32)
    zp = rng.integers(0, 16, size=(nb, 16, Hk), dtype=np.uint32)
    vs = (scale.view(np.uint32) & np.uint32(0xFFFFFFF0)) | zp
    q = bf16_inputs(rng, (B, Hq, D))
    signs = np.where(rng.random(D) < 0.5, F32(-1.0), F32(1.0)).astype(F32)
    sm = 1.0 / math.sqrt(D)
    out_rot = int4_cache.decode_int4(q, kc, vc, ks, vs, bt, lens, signs, sm)
    out_plain = int4_cache.decode_int4(q, kc, vc, ks, vs, bt, lens, None, sm)
    return {"B": B, "Hq": Hq, "Hk": Hk, "D": D, "num_blocks": nb, "seq_lens": lens.tolist(),
            "block_table": bt.tolist(), "k_cache": hexs(kc), "v_cache": hexs(vc), "k_scale": hexs(ks),
            "v_scale": hexs(vs), "q_bf16_as_f32": hexs(q), "signs": hexs(signs), "softmax_scale": sm,
            "out_rotated_f64": hexs(out_rot), "out_plain_f64": hexs(out_plain)}


def fwht_fixture(rng):
    x = bf16_inputs(rng, (4, 128))
    x[1] *= F32(1e-3)       # small row: the 1e-4 absmax floor is not reached, scale < 1
    x[2] = F32(0.0)         # all-zero row: absmax floored at 1e-4
    x[3, 7] = F32(3000.0)   # outlier row
    x = formats.bf16_round(x)  # the kernel's input is bf16: keep every fixture row bf16-exact
    y, s = fwht_fp8.fwht128_quant_fp8(x)
    return {"x_bf16_as_f32": hexs(x), "y_e4m3": hexs(y), "row_scale_f32": hexs(s)}


def tq_fixture(rng):
    Hk, D, G = 2, 128, 2
    out = {"Hk": Hk, "D": D, "Hq": Hk * G}
    for bits in (4, 3):
        vdb = turboquant.value_data_bytes(D, bits)
        slot = (D + vdb + 4 + 15) // 16 * 16
        cache = rng.integers(0, 256, size=(1, 16, Hk, slot), dtype=np.uint8)
        keys = formats.f32_to_e4m3fn(rng.standard_normal((16, Hk, D)).astype(F32))
        cache[0, :, :, :D] = keys
        sc = (rng.random((16, Hk)) * 0.2 + 0.01).astype(np.float16)
        ze = (rng.standard_normal((16, Hk)) * 0.5).astype(np.float16)
        cache[0, :, :, D + vdb:D + vdb + 2] = sc.view(np.uint8).reshape(16, Hk, 2)
        cache[0, :, :, D + vdb + 2:D + vdb + 4] = ze.view(np.uint8).reshape(16, Hk, 2)
        q = rng.standard_normal((1, Hk * G, D)).astype(F32)
        bt = np.array([[0]], dtype=np.int32)
        lens = np.array([13], dtype=np.int64)
        o = turboquant.decode_tq(q, cache, bits, bt, lens, 1.0 / math.sqrt(D))
        out["v%d" % bits] = {"slot_bytes": slot, "kv_cache": hexs(cache), "q_f32": hexs(q), "seq_len": 13,
                             "attn_scale": 1.0 / math.sqrt(D), "out_f64": hexs(o)}
    return out


def main():
    rng = np.random.default_rng(20261202)
    fixtures = {"int4_write_tiny.json": write_fixture(rng), "int4_decode_tiny.json": decode_fixture(rng),
                "fwht128_fp8_tiny.json": fwht_fixture(rng), "tq_decode_tiny.json": tq_fixture(rng)}
    for name, data in fixtures.items():
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)
            f.write("\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
