"""kvq_decode_int4 on the GPU against the float64 oracle on the same (oracle-written) cache.

Tolerance: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise (fp32 accumulation against the
float64 definition on the identical dequantized cache)."""

import math

import numpy as np
import pytest
import torch

from oracle import int4_cache
from quantized_paged_kv_int4_gb300 import kvq, workloads

from helpers import Int4Case, assert_close, run_int4

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num_splits", [4, 0, 1, 3, 7])
def test_tiny_config(num_splits):
    """B=2, Hq=4, Hk=2, D=64, seq_lens {37, 100}: ragged last pages, 4 warps per kv head."""
    c = Int4Case(workloads.tiny_int4())
    got = run_int4(kvq, c.to_gpu(), c.scale, num_splits=num_splits).cpu().numpy()
    assert_close(got, c.oracle(), what="tiny S=%d" % num_splits)


@pytest.mark.parametrize("Hk,G,D", [(1, 1, 128), (1, 8, 128), (2, 3, 64), (4, 2, 128), (8, 4, 128),
                                    (8, 8, 128), (16, 2, 64), (16, 5, 128), (8, 7, 64)])
def test_head_layouts(Hk, G, D):
    lens = [1, 15, 16, 17, 200, 513, 0, 33]
    case = workloads.DecodeCase("heads", len(lens), Hk * G, Hk, D, lens, seed=Hk * 10 + G, outlier_channels=4)
    c = Int4Case(case, num_blocks=sum(workloads.pages_needed(lens)) + 5)
    g = c.to_gpu()
    ref = c.oracle()
    for S in (0, 5):
        got = run_int4(kvq, g, c.scale, num_splits=S).cpu().numpy()
        assert_close(got, ref, what="Hk=%d G=%d D=%d S=%d" % (Hk, G, D, S))
        assert np.all(got[6] == 0.0)  # empty sequence


def test_unrotated_cache_and_output_dtypes():
    case = workloads.DecodeCase("norot", 3, 8, 2, 128, [77, 300, 5], seed=9)
    c = Int4Case(case, signs=False)
    g = c.to_gpu()
    ref = c.oracle()
    assert_close(run_int4(kvq, g, c.scale).cpu().numpy(), ref, what="f32")
    for dt in (torch.bfloat16, torch.float16):
        got = run_int4(kvq, g, c.scale, out_dtype=dt).float().cpu().numpy()
        assert_close(got, ref, atol=2e-3 + 1e-2, rtol=1e-2, what=str(dt))


def test_peaky_softmax():
    """A 30x larger softmax scale makes the distribution sharp: tests the running max rescale."""
    case = workloads.DecodeCase("peaky", 4, 32, 8, 128, [1000, 64, 4000, 17], seed=11, outlier_channels=4)
    c = Int4Case(case, scale_mult=30.0)
    got = run_int4(kvq, c.to_gpu(), c.scale).cpu().numpy()
    assert_close(got, c.oracle(), what="peaky")


def test_many_short_sequences_balanced():
    """More sequences than CTAs: a CTA's page run crosses many sequence boundaries."""
    rng = np.random.default_rng(12)
    lens = rng.integers(0, 60, size=700).tolist()
    case = workloads.DecodeCase("short", len(lens), 8, 2, 64, lens, seed=12)
    c = Int4Case(case, random_cache=True)
    got = run_int4(kvq, c.to_gpu(), c.scale).cpu().numpy()
    idx = list(range(0, 700, 37)) + [699]
    ref = c.oracle(batch_index=idx)
    assert_close(got[idx], ref[idx], what="short seqs")


def test_llama8b_decode_full_size_sampled():
    """B=32, Hq=32, Hk=8, D=128, seq_lens ~ U[1024, 8192]: the benchmark's launch (heuristic
    splits) on the full workload with a random cache; the oracle checks sampled sequences."""
    case = workloads.llama8b_int4()
    c = Int4Case(case, random_cache=True)
    g = c.to_gpu()
    got = run_int4(kvq, g, c.scale).cpu().numpy()
    idx = [0, 13, 31]
    ref = c.oracle(batch_index=idx)
    assert_close(got[idx], ref[idx], what="llama8b")
    assert np.all(np.isfinite(got))


def test_llama8b_decode_oracle_written_cache_medium():
    """Same shape family with the oracle writing the cache from K (4 outlier channels x10) and V."""
    case = workloads.DecodeCase("llama_med", 6, 32, 8, 128, [1024, 1500, 2049, 777, 3000, 1], seed=1,
                                outlier_channels=4)
    c = Int4Case(case)
    g = c.to_gpu()
    ref = c.oracle()
    for S in (0, 16):
        assert_close(run_int4(kvq, g, c.scale, num_splits=S).cpu().numpy(), ref, what="S=%d" % S)


def test_long_context_40gb_pool_sampled():
    """B=4, Hq=64, Hk=8, D=128, 131072 positions each, 64 splits, pages scattered in a 40 GB pool."""
    case = workloads.long_context_int4()
    Hk, D = case.Hk, case.D
    nb = case.pool_bytes // (16 * Hk * (D + 8))
    bt, _ = workloads.paged_layout(case.seq_lens, case.seed, num_blocks=nb)
    used = torch.unique(bt.flatten().to(torch.int64))
    dev = "cuda"
    kc = torch.empty((nb, 16, Hk, D // 2), dtype=torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    ks = torch.empty((nb, 16, Hk), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    kb, vb, kw, vw = workloads.random_int4_pages(used.numel(), Hk, D, case.seed)
    u = used.to(dev)
    kc[u] = kb.to(dev)
    vc[u] = vb.to(dev)
    ks[u] = kw.to(dev).view(torch.float32)
    vs[u] = vw.to(dev).view(torch.float32)
    q = workloads.query(case)
    signs = workloads.rht_signs(D)
    scale = 1.0 / math.sqrt(D)
    lens = torch.tensor(case.seq_lens, dtype=torch.int32)
    g = dict(q=q.to(dev), kc=kc, vc=vc, ks=ks, vs=vs, bt=bt.to(dev), lens=lens.to(dev), signs=signs.to(dev))
    # oracle on one sequence, reading only its pages (mapped into a compact pool)
    b = 2
    small_bt = np.zeros_like(bt.numpy())
    small_bt[b] = torch.searchsorted(used, bt[b].to(torch.int64)).numpy()
    ref = int4_cache.decode_int4(workloads.to_numpy_f32(q), kb.numpy(), vb.numpy(),
                                 kw.numpy().view(np.uint32), vw.numpy().view(np.uint32), small_bt,
                                 np.asarray(case.seq_lens), signs.numpy(), scale, batch_index=[b])
    for S in (64, 0):
        got = run_int4(kvq, g, scale, num_splits=S).cpu().numpy()
        assert_close(got[b], ref[b], what="long S=%d" % S)
    del kc, vc, ks, vs
    torch.cuda.empty_cache()


def test_workspace_reused_across_calls():
    """One workspace serves consecutive calls with identical results."""
    case = workloads.DecodeCase("reuse", 5, 16, 4, 128, [700, 1, 0, 2000, 333], seed=21, outlier_channels=4)
    c = Int4Case(case)
    g = c.to_gpu()
    ref = c.oracle()
    for S in (0, 6):
        ws = kvq.decode_workspace(case.B, case.Hq, case.Hk, case.D, S, device="cuda")
        outs = []
        for _ in range(3):
            o = kvq.kvq_decode_int4(g["q"], g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"],
                                    c.scale, workspace=ws, num_splits=S)
            outs.append(o.cpu().numpy())
        assert kvq.kvq_device_error() == (0, 0)
        assert_close(outs[0], ref, what="reuse S=%d" % S)
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


@pytest.mark.parametrize("num_splits", [0, 3])
def test_garbage_in_unwritten_rows_is_ignored(num_splits):
    """Rows of a sequence's last page past its length were never written: NaN scale words and
    arbitrary nibbles there must not reach the output."""
    case = workloads.DecodeCase("garbage", 4, 16, 4, 128, [37, 16, 250, 1], seed=31, outlier_channels=4)
    c = Int4Case(case)
    ref = c.oracle()
    nan_bits = np.uint32(0x7FC00000)
    for b, L in enumerate(case.seq_lens):
        page = int(c.bt[b, (L - 1) // 16])
        for row in range(L % 16 if L % 16 else 16, 16):
            c.ks[page, row] = nan_bits
            c.vs[page, row] = nan_bits
            c.kc[page, row] = 0xFF
            c.vc[page, row] = 0x5A
    got = run_int4(kvq, c.to_gpu(), c.scale, num_splits=num_splits).cpu().numpy()
    assert np.all(np.isfinite(got))
    assert_close(got, ref, what="garbage S=%d" % num_splits)


def test_prepared_writer_and_decoder_match_the_oracle():
    """Int4Writer / Int4Decoder (buffers checked once, per-step tensors per call) write the same
    bytes and decode the same rows as the oracle; wrong per-call shapes are rejected before launch."""
    case = workloads.DecodeCase("prep", 4, 32, 8, 128, [100, 1, 2049, 700], seed=71, outlier_channels=4)
    c = Int4Case(case)
    g = c.to_gpu()
    dec = kvq.Int4Decoder(g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale, case.Hq)
    out = torch.empty((4, 32, 128), dtype=torch.float32, device="cuda")
    for _ in range(2):
        dec(g["q"], out)
        assert kvq.kvq_device_error() == (0, 0)
        assert_close(out.cpu().numpy(), c.oracle(), what="prepared decoder")
    with pytest.raises(ValueError):
        dec(g["q"][:2], out)
    with pytest.raises(ValueError):
        dec(g["q"], out[:, :16])
    k, v, slots, nb = workloads.write_case(T=300, Hk=8, D=128, seed=3)
    kc = torch.zeros((nb, 16, 8, 64), dtype=torch.uint8, device="cuda")
    caches = [kc, torch.zeros_like(kc), torch.zeros((nb, 16, 8), device="cuda"), torch.zeros((nb, 16, 8), device="cuda")]
    ref = [t.clone() for t in caches]
    signs = workloads.rht_signs(128).cuda()
    kvq.Int4Writer(*caches, signs)(k.cuda(), v.cuda(), slots.cuda())
    kvq.kvq_write_int4(k.cuda(), v.cuda(), *ref, slots.cuda(), signs)
    for a, b in zip(caches, ref):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    with pytest.raises(ValueError):
        kvq.Int4Writer(*caches, signs)(k.cuda()[:, :4], v.cuda()[:, :4], slots.cuda())


def test_captured_step_replays_with_new_inputs():
    """kvq.CapturedStep: a step of (host-to-device copy of a staging buffer, decode, copy back)
    captured once and replayed with new staging contents gives, every replay, the oracle's rows for
    those contents and the same bytes as an eager call."""
    case = workloads.DecodeCase("graph", 3, 32, 8, 128, [300, 17, 1500], seed=72, outlier_channels=4)
    c = Int4Case(case)
    g = c.to_gpu()
    stream = torch.cuda.Stream()
    q_host = torch.empty(g["q"].shape, dtype=torch.bfloat16).pin_memory()
    q_dev = torch.empty_like(g["q"])
    out_dev = torch.empty((3, 32, 128), dtype=torch.float32, device="cuda")
    out_host = torch.empty(out_dev.shape, dtype=torch.float32).pin_memory()
    dec = kvq.Int4Decoder(g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"], c.scale, case.Hq)

    def calls():
        q_dev.copy_(q_host, non_blocking=True)
        dec(q_dev, out_dev, stream=stream)
        out_host.copy_(out_dev, non_blocking=True)

    q_host.copy_(g["q"].cpu())
    step = kvq.CapturedStep(calls, stream)
    for seed in (0, 1, 2):
        q_new = torch.randn(g["q"].shape, generator=torch.Generator().manual_seed(100 + seed)).to(torch.bfloat16)
        q_host.copy_(q_new)
        step()
        stream.synchronize()
        got = out_host.numpy().copy()
        c.q = q_new
        assert_close(got, c.oracle(), what="captured step, query set %d" % seed)
        eager = torch.empty_like(out_dev)
        kvq.kvq_decode_int4(q_new.cuda(), g["kc"], g["vc"], g["ks"], g["vs"], g["bt"], g["lens"], g["signs"],
                            c.scale, out=eager)
        assert np.array_equal(got, eager.cpu().numpy())
    assert kvq.kvq_device_error() == (0, 0)
