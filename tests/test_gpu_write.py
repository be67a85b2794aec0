"""kvq_write_int4 on the GPU against the oracle: every cache byte and scale word bit-exact."""

import numpy as np
import pytest
import torch

from oracle import int4_cache
from quantized_paged_kv_int4_gb300 import kvq, workloads

pytestmark = pytest.mark.gpu


def _write_both(k, v, slots, nb, Hk, D, signs, k_view=None, v_view=None):
    """Run the oracle and the GPU on the same inputs into sentinel-filled caches; compare all bytes."""
    kc = np.full((nb, 16, Hk, D // 2), 0xA5, np.uint8)
    vc = np.full((nb, 16, Hk, D // 2), 0x3C, np.uint8)
    ks = np.full((nb, 16, Hk), 0x7FC0DEAD, np.uint32)
    vs = np.full((nb, 16, Hk), 0x12345678, np.uint32)
    g = dict(kc=torch.from_numpy(kc).cuda(), vc=torch.from_numpy(vc).cuda(),
             ks=torch.from_numpy(ks.view(np.int32)).cuda().view(torch.float32),
             vs=torch.from_numpy(vs.view(np.int32)).cuda().view(torch.float32))
    int4_cache.write_int4(workloads.to_numpy_f32(k), workloads.to_numpy_f32(v), slots.numpy(),
                          None if signs is None else signs.numpy(), kc, vc, ks, vs)
    kk = k.cuda() if k_view is None else k_view
    vv = v.cuda() if v_view is None else v_view
    kvq.kvq_write_int4(kk, vv, g["kc"], g["vc"], g["ks"], g["vs"], slots.cuda(),
                       None if signs is None else signs.cuda())
    st, flags = kvq.kvq_device_error()
    assert st == 0 and flags == 0
    assert np.array_equal(g["kc"].cpu().numpy(), kc)
    assert np.array_equal(g["vc"].cpu().numpy(), vc)
    assert np.array_equal(g["ks"].cpu().view(torch.int32).numpy().view(np.uint32), ks)
    assert np.array_equal(g["vs"].cpu().view(torch.int32).numpy().view(np.uint32), vs)


@pytest.mark.parametrize("signs", [True, False])
def test_tiny_config_write(signs):
    case = workloads.tiny_int4()
    bt, nb = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=13)
    _, _, slots = workloads.all_token_slots(bt, case.seq_lens)
    k, v = workloads.kv_vectors(case, slots.numel())
    slots = slots.clone()
    slots[::5] = -1
    _write_both(k, v, slots, nb, case.Hk, case.D, workloads.rht_signs(case.D) if signs else None)


def test_full_write_workload_16384_tokens():
    """16384 new tokens x 8 heads x 128, 5 % holes in slot_mapping, pages of 16."""
    k, v, slots, nb = workloads.write_case()
    _write_both(k, v, slots, nb, 8, 128, workloads.rht_signs(128))


def test_strided_views_and_special_rows():
    """K and V as strided views of a fused QKV tensor; constant, zero and huge rows."""
    T, Hk, D, Hq = 300, 4, 128, 16
    qkv = workloads.bf16_normal((T, Hq + 2 * Hk, D), seed=3, k=2)
    qkv[0, Hq] = 10.0                     # constant row
    qkv[1, Hq:Hq + Hk] = 0.0              # zero rows (scale floor 1e-6)
    qkv[2, Hq] = 3000.0                   # float -> int saturation without rotation
    qkv[3, Hq, :64] = -2.0e4
    kv_gpu = qkv.cuda()
    kk = kv_gpu[:, Hq:Hq + Hk]
    vv = kv_gpu[:, Hq + Hk:]
    assert kk.stride(0) == (Hq + 2 * Hk) * D and not kk.is_contiguous()
    nb = T // 16 + 3
    slots = torch.randperm(nb * 16, generator=torch.Generator().manual_seed(4))[:T].to(torch.int64)
    k = qkv[:, Hq:Hq + Hk].contiguous()
    v = qkv[:, Hq + Hk:].contiguous()
    for signs in (workloads.rht_signs(D), None):
        _write_both(k, v, slots, nb, Hk, D, signs, k_view=kk, v_view=vv)


def test_empty_and_all_skipped():
    k, v, slots, nb = workloads.write_case(T=64, Hk=2, D=64, hole_frac=1.01)
    assert (slots < 0).all()
    _write_both(k, v, slots, nb, 2, 64, workloads.rht_signs(64))
    kc = torch.zeros((4, 16, 2, 32), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((4, 16, 2), dtype=torch.float32, device="cuda")
    e = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    kvq.kvq_write_int4(e, e, kc, kc, sc, sc, torch.empty((0,), dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()


@pytest.mark.parametrize("Hk,D,T", [(1, 64, 777), (3, 128, 777), (5, 64, 1001), (12, 128, 301), (12, 128, 2049),
                                    (24, 64, 341), (6, 128, 1365), (6, 128, 1366)])
def test_head_counts_and_ragged_tiles(Hk, D, T):
    """Head counts that are not powers of two (the kernels split a pair index into token and head
    by a multiply-shift) and pair counts that leave a ragged last tile of 16 pairs; writes of up to
    8192 (token, head) pairs take the eight-lanes-per-vector kernel, larger ones the one-thread-per-
    vector kernel (6 x 1365 = 8190 pairs sit just below the switch, 6 x 1366 = 8196 just above)."""
    k, v, slots, nb = workloads.write_case(T=T, Hk=Hk, D=D, hole_frac=0.1, seed=Hk)
    _write_both(k, v, slots, nb, Hk, D, workloads.rht_signs(D))


def test_many_tiles_per_cta():
    """More 16-pair tiles than resident CTAs: every CTA walks several tiles with the next one's
    rows fetched ahead (65536 tokens x 3 heads = 12288 tiles)."""
    k, v, slots, nb = workloads.write_case(T=65536, Hk=3, D=64, hole_frac=0.02, seed=11)
    _write_both(k, v, slots, nb, 3, 64, None)
