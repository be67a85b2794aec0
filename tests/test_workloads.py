"""The seeded input generators shared by the oracle, the tests and the bench (CPU): they are
deterministic per seed, the page tables they build are valid (every physical page used once, in
range, padded past each sequence), the token slots address the right pages, and the layout
helpers agree with the byte counts they describe."""

import numpy as np
import pytest
import torch

from quantized_paged_kv_int4_gb300 import workloads


def _same(a, b):
    if isinstance(a, torch.Tensor):
        return torch.equal(a, b)
    if isinstance(a, (tuple, list)):
        return len(a) == len(b) and all(_same(x, y) for x, y in zip(a, b))
    return a == b


@pytest.mark.parametrize("make", [
    lambda s: workloads.paged_layout([37, 100, 0, 16], s),
    lambda s: workloads.paged_layout([37, 100, 5], s, num_blocks=1000, unused_fill=-1),
    lambda s: workloads.bf16_normal((4, 8, 64), s, 2),
    lambda s: workloads.fwht_rows(rows=64, seed=s),
    lambda s: workloads.random_rotation(64, s),
    lambda s: workloads.random_int4_pages(3, 2, 64, s),
    lambda s: workloads.kpool_case(8, 4, 16, seed=s),
])
def test_generators_are_deterministic_per_seed(make):
    a, b, c = make(3), make(3), make(4)
    assert _same(a, b)
    assert not _same(a, c)


@pytest.mark.parametrize("num_blocks", [None, 5000])
def test_paged_layout_is_a_valid_page_table(num_blocks):
    lens = [37, 100, 0, 16, 1, 4096]
    bt, nb = workloads.paged_layout(lens, 7, num_blocks=num_blocks, unused_fill=-1)
    need = workloads.pages_needed(lens)
    assert need == [-(-L // 16) for L in lens]
    assert bt.dtype == torch.int32 and bt.shape == (len(lens), max(need))
    used = []
    for b, n in enumerate(need):
        row = bt[b].tolist()
        used += row[:n]
        assert all(x == -1 for x in row[n:])          # padding past the sequence's last page
    assert len(used) == len(set(used)) == sum(need)   # every physical page at most once
    assert all(0 <= x < nb for x in used)
    if num_blocks is None:
        assert nb == sum(need) and sorted(used) == list(range(nb))


def test_token_slots_address_their_pages():
    lens = [37, 100, 16]
    bt, nb = workloads.paged_layout(lens, 1)
    seq, pos, slots = workloads.all_token_slots(bt, lens)
    assert slots.numel() == sum(lens) and len(set(slots.tolist())) == sum(lens)
    for s, p, x in zip(seq.tolist(), pos.tolist(), slots.tolist()):
        assert x // 16 == int(bt[s, p // 16]) and x % 16 == p % 16
    pick = workloads.slots_for_positions(bt, 1, torch.tensor([0, 15, 16, 99]))
    assert pick.tolist() == [int(bt[1, 0]) * 16, int(bt[1, 0]) * 16 + 15, int(bt[1, 1]) * 16,
                             int(bt[1, 6]) * 16 + 3]


def test_rht_signs_are_plus_minus_one_and_seeded_by_round():
    s0, s0b, s1 = workloads.rht_signs(128), workloads.rht_signs(128), workloads.rht_signs(128, 1)
    assert set(s0.tolist()) <= {-1.0, 1.0} and torch.equal(s0, s0b) and not torch.equal(s0, s1)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kb,vb", [(3, 4), (4, 4), (3, 3), (4, 3)])
def test_mse_layout_byte_counts(D, kb, vb):
    mse, kps, sb = workloads.turboquant_mse_layout(D, kb, vb)
    assert mse * 8 >= D * kb > (mse - 1) * 8        # whole index stream, no spare byte
    assert kps == mse + 2                            # the fp16 norm right after the indices
    vdb = -(-D * vb // 8)
    assert sb % 16 == 0 and kps + vdb + 4 <= sb < kps + vdb + 4 + 16
    cb = workloads.mse_codebook(kb, D)
    assert cb.shape == (1 << kb,) and torch.all(cb[1:] > cb[:-1])
    assert torch.allclose(cb, -cb.flip(0), atol=1e-7)  # quantiles symmetric about zero


def test_random_rotation_is_orthogonal():
    P = workloads.random_rotation(128, 2).double()
    assert P.is_contiguous()
    assert torch.allclose(P @ P.T, torch.eye(128, dtype=torch.float64), atol=1e-5)
