"""The C ABI without a GPU: the library builds and loads, exports every symbol include/kvq.h
declares, and host-side validation rejects bad arguments before anything is launched.

Every call below is one that validation rejects (or an empty no-op): none reaches a launch, so
the fake pointers are never used."""

import ctypes
import os
import re

import pytest

from quantized_paged_kv_int4_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", text)


def test_header_declares_the_api():
    names = _declared()
    assert sorted(names) == sorted(kvq.C_FUNCTIONS)


def test_library_exports_every_declared_symbol():
    h = ctypes.CDLL(kvq.lib()._name)
    for name in _declared():
        assert hasattr(h, name), name


def test_status_strings_and_version():
    assert kvq.kvq_abi_version() == 5
    for code in range(6):
        assert kvq.kvq_status_string(code).startswith("KVQ_")
    assert "UNKNOWN" in kvq.kvq_status_string(77)


def _write(**kw):
    args = dict(key=16, value=16, kst=1024, ksh=128, vst=1024, vsh=128, kc=16, vc=16, ks=16, vs=16, slots=16,
                signs=None, T=4, Hk=8, D=128, bs=16, nb=10, stream=None)
    args.update(kw)
    L = kvq.lib()
    return L.kvq_write_int4(args["key"], args["value"], args["kst"], args["ksh"], args["vst"], args["vsh"],
                            args["kc"], args["vc"], args["ks"], args["vs"], args["slots"], args["signs"],
                            args["T"], args["Hk"], args["D"], args["bs"], args["nb"], args["stream"])


def test_write_validation_without_gpu():
    assert _write(T=0) == kvq.KVQ_OK                      # empty: no-op
    assert _write(D=96) == kvq.KVQ_ERR_UNSUPPORTED
    assert _write(key=None) == kvq.KVQ_ERR_INVALID_ARG
    assert _write(key=17) == kvq.KVQ_ERR_INVALID_ARG      # misaligned
    assert _write(kst=1001) == kvq.KVQ_ERR_INVALID_ARG    # stride not a vector multiple
    assert _write(Hk=0) == kvq.KVQ_ERR_INVALID_ARG
    assert _write(nb=0) == kvq.KVQ_ERR_INVALID_ARG
    assert _write(T=-1) == kvq.KVQ_ERR_INVALID_ARG


def _decode(**kw):
    a = dict(q=16, kc=16, vc=16, ks=16, vs=16, bt=16, mb=4, sl=16, signs=None, scale=0.1, S=4, ws=16,
             wsb=1 << 30, out=16, od=kvq.KVQ_F32, B=2, Hq=4, Hk=2, D=64, bs=16, nb=10, stream=None)
    a.update(kw)
    return kvq.lib().kvq_decode_int4(a["q"], a["kc"], a["vc"], a["ks"], a["vs"], a["bt"], a["mb"], a["sl"],
                                     a["signs"], a["scale"], a["S"], a["ws"], a["wsb"], a["out"], a["od"],
                                     a["B"], a["Hq"], a["Hk"], a["D"], a["bs"], a["nb"], a["stream"])


def test_decode_validation_without_gpu():
    assert _decode(B=0) == kvq.KVQ_OK
    assert _decode(D=80) == kvq.KVQ_ERR_UNSUPPORTED
    assert _decode(bs=32) == kvq.KVQ_ERR_UNSUPPORTED
    assert _decode(Hq=36, Hk=2) == kvq.KVQ_ERR_UNSUPPORTED     # 18 query heads per kv head
    assert _decode(Hk=3, Hq=6) == kvq.KVQ_ERR_UNSUPPORTED      # kv heads not a power of two <= 8
    assert _decode(Hq=5) == kvq.KVQ_ERR_INVALID_ARG            # Hq % Hk
    assert _decode(scale=0.0) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode(q=None) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode(out=20) == kvq.KVQ_ERR_INVALID_ARG          # misaligned output
    assert _decode(od=7) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode(wsb=10) == kvq.KVQ_ERR_WORKSPACE


def _decode_mods(mods, **kw):
    a = dict(q=16, kc=16, vc=16, ks=16, vs=16, bt=16, mb=4, sl=16, signs=None, scale=0.1, S=4, ws=16,
             wsb=1 << 30, out=16, od=kvq.KVQ_F32, B=2, Hq=4, Hk=2, D=64, bs=16, nb=10, stream=None)
    a.update(kw)
    return kvq.lib().kvq_decode_int4_mods(a["q"], a["kc"], a["vc"], a["ks"], a["vs"], a["bt"], a["mb"], a["sl"],
                                          a["signs"], a["scale"], a["S"], a["ws"], a["wsb"], a["out"], a["od"],
                                          a["B"], a["Hq"], a["Hk"], a["D"], a["bs"], a["nb"],
                                          None if mods is None else ctypes.byref(mods), a["stream"])


def test_decode_mods_validation_without_gpu():
    M = kvq.ScoreMods
    assert _decode_mods(None, B=0) == kvq.KVQ_OK
    assert _decode_mods(M(0, 0.0, None, None), B=0) == kvq.KVQ_OK
    assert _decode_mods(M(-1, 0.0, None, None)) == kvq.KVQ_ERR_INVALID_ARG       # negative window
    assert _decode_mods(M(0, -1.0, None, None)) == kvq.KVQ_ERR_INVALID_ARG       # negative cap
    assert _decode_mods(M(0, float("inf"), None, None)) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode_mods(M(0, float("nan"), None, None)) == kvq.KVQ_ERR_INVALID_ARG
    assert _decode_mods(M(0, 0.0, 18, None)) == kvq.KVQ_ERR_INVALID_ARG          # misaligned sinks
    assert _decode_mods(M(0, 0.0, None, 18)) == kvq.KVQ_ERR_INVALID_ARG          # misaligned slopes
    assert _decode_mods(M(8, 30.0, 16, 16), wsb=10) == kvq.KVQ_ERR_WORKSPACE      # then the usual checks
    assert _decode_mods(M(0, 0.0, None, None, 1, 18)) == kvq.KVQ_ERR_INVALID_ARG  # misaligned lse_out
    assert _decode_mods(M(0, 0.0, None, None, 1, 16), B=0) == kvq.KVQ_OK


def test_workspace_sizes_fixed_splits():
    # fixed splits need no device query: slots = B * S, 8 / Hk warps per head, Hq rows of D + lse,
    # then the first / last CTA of each sequence, then the single-token INT4 call's rotated query
    # fragments (2 D/16 + 3 words for each of 32 lanes per (sequence, kv head))
    n = kvq.kvq_decode_workspace_bytes(2, 4, 2, 64, 4)
    rows = 2 * 4 * 4 * 4
    r256 = lambda x: (x + 255) // 256 * 256
    frag = lambda B, Hk, D: r256(B * Hk * (2 * (D // 16) + 3) * 32 * 4)
    assert n == r256(rows * 64 * 4) + r256(rows * 4) + 2 * r256(2 * 4) + frag(2, 2, 64)
    n16 = kvq.kvq_decode_workspace_bytes(3, 32, 16, 128, 2)   # 2 head groups of 8 kv heads
    rows = 3 * 2 * 1 * 32
    assert n16 == r256(rows * 128 * 4) + r256(rows * 4) + 2 * r256(3 * 4) + frag(3, 16, 128)
    assert kvq.kvq_decode_workspace_bytes(2, 4, 2, 80, 4) == 0
    assert kvq.kvq_decode_workspace_bytes(2, 4, 3, 64, 4) == 0


def test_tq_and_fwht_validation_without_gpu():
    L = kvq.lib()
    args = [16, 16, 208, 4, 16, 4, 16, ctypes.c_float(0.1), 4, 16, 1 << 30, 16, 2, 4, 2, 128, 16, 10, None]
    bad = list(args)
    bad[3] = 5
    assert L.kvq_decode_tq(*bad) == kvq.KVQ_ERR_UNSUPPORTED       # value bits
    bad = list(args)
    bad[2] = 200
    assert L.kvq_decode_tq(*bad) == kvq.KVQ_ERR_INVALID_ARG       # slot not a multiple of 16
    bad = list(args)
    bad[2] = 192
    assert L.kvq_decode_tq(*bad) == kvq.KVQ_ERR_INVALID_ARG       # too small for 4-bit values
    bad = list(args)
    bad[12] = 0
    assert L.kvq_decode_tq(*bad) == kvq.KVQ_OK                    # B = 0
    lse = list(args[:12]) + [18] + list(args[12:])
    assert L.kvq_decode_tq_lse(*lse) == kvq.KVQ_ERR_INVALID_ARG   # misaligned lse_out
    lse[3] = 5
    assert L.kvq_decode_tq_lse(*lse) == kvq.KVQ_ERR_UNSUPPORTED   # the usual checks come first (value bits)
    lse = list(args[:12]) + [None] + list(args[12:])
    lse[13] = 0
    assert L.kvq_decode_tq_lse(*lse) == kvq.KVQ_OK                # B = 0
    assert L.kvq_fwht128(16, 16, 16, 0, None) == kvq.KVQ_OK
    assert L.kvq_fwht128(18, 16, 16, 5, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_fwht128(16, 16, 16, -1, None) == kvq.KVQ_ERR_INVALID_ARG


def test_tq_mse_validation_without_gpu():
    L = kvq.lib()
    # q, Pi, centroids, cache, slot 128, key 3, kps 50, value 4, norm corr, bt, mb, lens, scale, S, ws, wsb,
    # out, B, Hq, Hk, D, bs, nb, stream
    args = [16, 16, 16, 16, 128, 3, 50, 4, 0, 16, 4, 16, ctypes.c_float(0.1), 4, 256, 1 << 30, 16, 2, 4, 2, 128,
            16, 10, None]
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.kvq_decode_tq_mse(*a)
    assert call(a17=0) == kvq.KVQ_OK                          # B = 0
    assert call(a5=5) == kvq.KVQ_ERR_UNSUPPORTED              # key bits
    assert call(a7=8) == kvq.KVQ_ERR_UNSUPPORTED              # value bits
    assert call(a6=49) == kvq.KVQ_ERR_INVALID_ARG             # kps odd / below MSE_BYTES + 2
    assert call(a6=48) == kvq.KVQ_ERR_INVALID_ARG
    assert call(a4=112) == kvq.KVQ_ERR_INVALID_ARG            # slot too small for the 4-bit values
    assert call(a4=130) == kvq.KVQ_ERR_INVALID_ARG            # not a multiple of 16
    assert call(a14=272) == kvq.KVQ_ERR_INVALID_ARG           # workspace not 256-byte aligned
    assert call(a15=100) == kvq.KVQ_ERR_WORKSPACE
    n = kvq.kvq_decode_tq_mse_workspace_bytes(2, 4, 2, 128, 4)
    int4_frag = 2 * 2 * (2 * (128 // 16) + 3) * 32 * 4  # the INT4 call's query fragments (not used here)
    assert n == kvq.kvq_decode_workspace_bytes(2, 4, 2, 128, 4) - int4_frag + 2 * 4 * 128 * 4


def test_kpool_validation_without_gpu():
    L = kvq.lib()
    args = [16, 16, 16, 16, 16, None, 8, 4, 128, 16, 10, 1, None]
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.kvq_kpool_write(*a)
    assert call(a6=0) == kvq.KVQ_OK                        # no pools
    assert call(a8=64) == kvq.KVQ_ERR_UNSUPPORTED          # head_dim
    assert call(a9=6) == kvq.KVQ_ERR_UNSUPPORTED           # page_size not a multiple of 4
    assert call(a7=0) == kvq.KVQ_ERR_INVALID_ARG           # pool_size
    assert call(a1=None) == kvq.KVQ_ERR_INVALID_ARG
    assert call(a2=20) == kvq.KVQ_ERR_INVALID_ARG          # misaligned scores
    assert call(a4=12) == kvq.KVQ_ERR_INVALID_ARG          # misaligned loc


def test_kpool_tail_validation_without_gpu():
    L = kvq.lib()
    # tail, block stride, half stride, ring, blocks, key, score, tslot, n, kpool, head_dim, stream
    seed = [16, 2 * 8 * 128, 8 * 128, 8, 4, 16, 16, 16, 5, 4, 128, None]
    def call(args, **kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return a
    assert L.kvq_kpool_seed_tail(*call(seed, a8=0)) == kvq.KVQ_OK
    assert L.kvq_kpool_seed_tail(*call(seed, a10=64)) == kvq.KVQ_ERR_UNSUPPORTED
    assert L.kvq_kpool_seed_tail(*call(seed, a1=100)) == kvq.KVQ_ERR_INVALID_ARG     # block stride too small
    assert L.kvq_kpool_seed_tail(*call(seed, a0=18)) == kvq.KVQ_ERR_INVALID_ARG      # misaligned tail
    upd = [16, 16, 10, 16, 2 * 8 * 128, 8 * 128, 8, 4, 16, 16, 3 * 128, 128, 16, 3 * 128, 128, 16, 16, 16, 2, 3, 4,
           128, 1, None]
    assert L.kvq_kpool_decode_update(*call(upd, a18=0)) == kvq.KVQ_OK                # no requests
    assert L.kvq_kpool_decode_update(*call(upd, a6=6)) == kvq.KVQ_ERR_INVALID_ARG    # ring % pool
    assert L.kvq_kpool_decode_update(*call(upd, a6=2)) == kvq.KVQ_ERR_INVALID_ARG    # ring < pool
    assert L.kvq_kpool_decode_update(*call(upd, a21=64)) == kvq.KVQ_ERR_UNSUPPORTED
    assert L.kvq_kpool_decode_update(*call(upd, a10=130)) == kvq.KVQ_ERR_INVALID_ARG  # key stride


@pytest.mark.parametrize("name", ["kvq_write_int4", "kvq_decode_int4", "kvq_decode_tq", "kvq_decode_tq_mse",
                                  "kvq_kpool_write", "kvq_kpool_seed_tail", "kvq_kpool_decode_update",
                                  "kvq_fwht128"])
def test_python_binding_names_match_the_c_api(name):
    assert callable(getattr(kvq, name))


def test_debug_wait_setting_without_gpu():
    L = kvq.lib()
    assert L.kvq_debug_set_wait(0, -2) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_debug_set_wait(0, -1) == kvq.KVQ_OK      # the defaults
