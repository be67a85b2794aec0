#!/usr/bin/env python
"""Benchmark of the INT4 paged decode step on GB300 (one JSON line on stdout).

Default workload (llama3_8b_int4): B=32, Hq=32, Hk=8, D=128, block 16, seq_lens ~ U[1024, 8192]
(seed 0), INT4 K/V with the random-sign Hadamard rotation. One step = the whole hot path of a
decode step: kvq_write_int4 of the B new tokens' K/V (position seq_len - 1 of each sequence) and
kvq_decode_int4 over the paged cache (q rotation, split-KV attention, log-sum-exp merge,
inverse rotation), bf16 output.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference] [--workload NAME]

Timing: each step replays CUDA graphs (write, decode) captured from the public API; the K timed
steps are bracketed by a barrier + synchronize and CUDA events on the launching stream. Four
independent cache replicas rotate between steps, so no step's inputs are still in L2 (the
working set is 4 x ~160 MB against a 126 MB L2). The decode call is also bracketed by its own
events every step (roofline). `e2e` repeats the step through the public API from pinned host
memory: one H2D copy of the step's inputs (staged in one pinned buffer), write + decode, D2H of
the output, synchronize, wall clock.
`--impl reference` times the CPU oracle (test infrastructure) on a bounded sample instead.
N > 1 (torchrun): every rank runs its own replica of the workload (no collective on the data
path); value = all ranks' bytes / max-over-ranks time.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_paged_kv_int4_gb300 import kvq, workloads  # noqa: E402

METRIC = "INT4 paged decode attention: KV-cache GB/s read (% HBM peak), µs per step"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default="llama3_8b_int4",
                    choices=["llama3_8b_int4", "llama3_8b_int4_mods", "llama3_8b_int4_q2", "long_context_int4",
                             "turboquant_fp8_v4",
                             "turboquant_fp8_v3", "turboquant_mse_k3v4", "write_fwht", "kpool_write",
                             "kpool_decode_update"])
    ap.add_argument("--replicas", type=int, default=4)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--burn-in-s", type=float, default=1.5)
    return ap.parse_args()


# ----------------------------------------------------------------------------------------------
# distributed plumbing (host-side only: barrier and max-over-ranks of the timings)
# ----------------------------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x):
        if not self.pg:
            return x
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x):
        if not self.pg:
            return x
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------------------------
# measured peaks, clocks, ncu traffic
# ----------------------------------------------------------------------------------------------
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def ncu_traffic(kernel_tag, source_files):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on the current sources."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[kernel_tag]
    except Exception:
        return None
    h = hashlib.sha256()
    for s in source_files:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    if rec.get("sources_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------------------------
def int4_decode_bytes(lens, Hq, Hk, D, out_bytes=2, window=0):
    """Algorithmic bytes of one decode call: the keys read (the last `window` of each sequence
    under a sliding window) at D + 8 bytes per (token, kv head), their block-table entries, q,
    out and seq_lens."""
    kv, bt = 0, 0
    for L in lens:
        lo = max(0, L - window) if window > 0 else 0
        kv += (L - lo) * Hk * (D + 8)
        bt += ((L - 1) // 16 - lo // 16 + 1) * 4 if L > 0 else 0
    return kv + bt + len(lens) * Hq * D * (2 + out_bytes) + 4 * len(lens), kv


class Int4Replica:
    """One independent copy of the decode-step inputs, resident in HBM.

    The cache is written by kvq_write_int4 from the workload's K / V recipe: K ~ N(0, 1) with the
    case's outlier channels x10 (applied before the rotation), V ~ N(0, 1), every position of every
    sequence at its block-table slot, drawn on the device from a seeded generator."""

    def __init__(self, case, seed, dev, signs, pool_blocks=None):
        B, Hq, Hk, D = case.B, case.Hq, case.Hk, case.D
        lens = case.seq_lens
        self.bt, self.nb = workloads.paged_layout(lens, seed, num_blocks=pool_blocks)
        nb = self.nb
        alloc = torch.empty if pool_blocks is not None else torch.zeros  # a 40 GB pool: only used pages written
        self.kc = alloc((nb, 16, Hk, D // 2), dtype=torch.uint8, device=dev)
        self.vc = alloc((nb, 16, Hk, D // 2), dtype=torch.uint8, device=dev)
        self.ks = alloc((nb, 16, Hk), dtype=torch.float32, device=dev)
        self.vs = alloc((nb, 16, Hk), dtype=torch.float32, device=dev)
        _, _, slots = workloads.all_token_slots(self.bt, lens)
        ch = workloads.outlier_channels(D, case.outlier_channels, case.seed).to(dev)
        g = torch.Generator(device=dev)
        g.manual_seed(1000 + seed)
        for lo in range(0, slots.numel(), 65536):
            sl = slots[lo:lo + 65536].to(dev)
            k = torch.randn((sl.numel(), Hk, D), generator=g, device=dev)
            if ch.numel():
                k[:, :, ch] *= case.outlier_scale
            v = torch.randn((sl.numel(), Hk, D), generator=g, device=dev)
            kvq.kvq_write_int4(k.to(torch.bfloat16), v.to(torch.bfloat16), self.kc, self.vc, self.ks, self.vs, sl,
                               signs)
        torch.cuda.synchronize(dev)
        self.bt = self.bt.to(dev)
        self.lens = torch.tensor(lens, dtype=torch.int32, device=dev)
        cpu = torch.Generator().manual_seed(2000 + seed)
        self.q = torch.randn((B, Hq, D), generator=cpu).to(torch.bfloat16).to(dev)
        self.k_new = torch.randn((B, Hk, D), generator=cpu).to(torch.bfloat16).to(dev)
        self.v_new = torch.randn((B, Hk, D), generator=cpu).to(torch.bfloat16).to(dev)
        last = torch.tensor([L - 1 for L in lens], dtype=torch.int64)
        self.slots = workloads.slots_for_positions(self.bt.cpu(), torch.arange(B), last).to(dev)
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)


def run_kvq(args, dist):
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    wl = args.workload
    if wl == "write_fwht":
        return run_write_fwht(args, dist, dev, stream)
    if wl == "kpool_write":
        return run_kpool(args, dist, dev, stream)
    if wl == "kpool_decode_update":
        return run_kpool_update(args, dist, dev, stream)
    if wl.startswith("turboquant_mse"):
        return run_tq_mse(args, dist, dev, stream)
    if wl.startswith("turboquant"):
        return run_tq(args, dist, dev, stream)
    case = workloads.long_context_int4() if wl == "long_context_int4" else workloads.llama8b_int4()
    B, Hq, Hk, D = case.B, case.Hq, case.Hk, case.D
    signs = workloads.rht_signs(D).to(dev)
    scale = 1.0 / math.sqrt(D)
    mods = {}
    if wl == "llama3_8b_int4_mods":  # every score modifier at once: 4096-key window, cap 30, ALiBi, sinks
        mods = dict(sliding_window=4096, softcap=30.0,
                    alibi_slopes=(2.0 ** (-8.0 * (torch.arange(Hq, dtype=torch.float32) + 1) / Hq)).to(dev),
                    sinks=(torch.randn((Hq,), generator=torch.Generator().manual_seed(5)) * 2.0).to(dev))
    pool = None
    nrep = args.replicas
    if wl == "long_context_int4":
        pool = case.pool_bytes // (16 * Hk * (D + 8))
        nrep = 1  # 570 MB read per step: far beyond L2 by itself
    reps = [Int4Replica(case, 10 * dist.rank + r, dev, signs, pool) for r in range(nrep)]
    S = case.num_splits
    ws = torch.zeros((kvq.kvq_decode_workspace_bytes(B, Hq, Hk, D, S),), dtype=torch.uint8, device=dev)

    def write(r):
        kvq.kvq_write_int4(r.k_new, r.v_new, r.kc, r.vc, r.ks, r.vs, r.slots, signs, stream=stream)

    Q = 2 if wl == "llama3_8b_int4_q2" else 1  # speculative verify: two query tokens per sequence
    if Q > 1:
        mods = dict(q_len=Q)
        gq = torch.Generator().manual_seed(77)
        for r in reps:
            r.q = torch.randn((B * Q, Hq, D), generator=gq).to(torch.bfloat16).to(dev)
            r.out = torch.empty((B * Q, Hq, D), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros((kvq.kvq_decode_int4_mods_workspace_bytes(B, Hq, Hk, D, S, kvq.ScoreMods(q_len=Q)),),
                         dtype=torch.uint8, device=dev)

    def decode(r):
        kvq.kvq_decode_int4(r.q, r.kc, r.vc, r.ks, r.vs, r.bt, r.lens, signs, scale, out=r.out, workspace=ws,
                            num_splits=S, stream=stream, **mods)

    with torch.cuda.stream(stream):
        for r in reps:  # eager warm-up (also sets kernel attributes before capture)
            write(r)
            decode(r)
    stream.synchronize()
    st, flags = kvq.kvq_device_error(stream)
    assert st == 0, flags
    gw, gd, gs = [], [], []  # per replica: the write, the decode, and the whole step (both) as one graph
    for r in reps:
        a, b, c = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(a, stream=stream):
            write(r)
        with torch.cuda.graph(b, stream=stream):
            decode(r)
        with torch.cuda.graph(c, stream=stream):
            write(r)
            decode(r)
        gw.append(a)
        gd.append(b)
        gs.append(c)

    dec_bytes, kv_bytes = int4_decode_bytes(case.seq_lens, Q * Hq, Hk, D, window=mods.get("sliding_window", 0))
    dec_bytes += 8 * Hq if "sinks" in mods else 0  # sinks and slopes
    wr_bytes = B * Hk * (2 * D * 2 + 2 * (D // 2 + 4)) + 8 * B
    res = timed_steps(args, dist, stream, lambda i: gw[i % nrep].replay(), lambda i: gd[i % nrep].replay(),
                      dev.index, step=lambda i: gs[i % nrep].replay())
    st, flags = kvq.kvq_device_error(stream)
    assert st == 0, flags

    e2e = None
    if not args.no_e2e and not mods and Q == 1:
        e2e = e2e_int4(args, reps[0], case, signs, scale, ws, S, dev, stream, dec_bytes)
    cfg = {"workload": wl, "B": B, "Hq": Hq, "Hk": Hk, "D": D, "block_size": 16,
           "seq_lens": "U[1024,8192] seed 0, sum %d" % sum(case.seq_lens) if wl != "long_context_int4"
           else "131072 x 4, pages scattered in a %.0f GB pool" % (case.pool_bytes / 1e9),
           "num_splits": "heuristic (balanced)" if S == 0 else S, "rht": True, "out_dtype": "bf16",
           "step": "kvq_write_int4 (B new tokens) + kvq_decode_int4, replayed as one CUDA graph",
           "l2": ("%d rotating cache replicas, %.0f MB read from each per step (%d x %.0f MB > 126 MB L2): "
                  "no L2 reuse across steps" % (nrep, kv_bytes / 1e6, nrep, kv_bytes / 1e6)) if nrep > 1
           else "single %.0f MB cache read per step (> L2)" % (kv_bytes / 1e6),
           "decode_bytes_per_step": dec_bytes, "kv_cache_bytes_per_step": kv_bytes, "write_bytes_per_step": wr_bytes}
    if Q > 1:
        cfg["q_len"] = "%d query tokens per sequence (causal; keys read once for both)" % Q
    if "sinks" in mods:
        cfg["score_mods"] = "sliding_window 4096 (keys read: %d of %d), softcap 30, ALiBi slopes 2^(-8(h+1)/Hq), sinks" % (
            kv_bytes // (Hk * (D + 8)), sum(case.seq_lens))
    # write, then the call's kernels: q rotation (plain single-token calls), virtual-sequence setup
    # (multi-token calls), split-KV decode, merge
    kernels = 3 + (1 if (not mods and Q == 1) or Q > 1 else 0)
    tag = {"llama3_8b_int4": "decode_int4", "long_context_int4": "decode_int4_long_context",
           "llama3_8b_int4_q2": "decode_int4_q2"}.get(wl, "decode_int4_mods")
    return finish(args, dist, res, dec_bytes, cfg, e2e, kernels, tag,
                  ["quantized_paged_kv_int4_gb300/csrc/decode_int4.cu",
                   "quantized_paged_kv_int4_gb300/csrc/decode_common.cuh",
                   "quantized_paged_kv_int4_gb300/csrc/kvq_device.cuh"], "f32")


def timed_steps(args, dist, stream, first, second, dev_index, step=None):
    """W warm-up steps, a burn-in (clock sampling), then the timed region: K steps back to back
    between one event pair (the step time); K `second` calls (the dominant call) back to back
    between one event pair (its average launch duration, nothing inside the region but the calls);
    and K more steps with an event pair around each `second` call (the same duration seen with
    an event on each side, which adds about 2 us per call; reported beside it). Clocks are
    sampled over all three. `step(i)`, when given, replays step i as one graph (first and second
    captured together) in the step-time pass."""
    if step is None:
        step = lambda i: (first(i), second(i))
    for i in range(args.warmup):
        with torch.cuda.stream(stream):
            step(i)
            first(i)
            second(i)
    stream.synchronize()
    sampler = ClockSampler(dev_index)
    sampler.start()
    t_end = time.perf_counter() + args.burn_in_s
    i = 0
    while time.perf_counter() < t_end:
        with torch.cuda.stream(stream):
            first(i)
            second(i)
        i += 1
        if i % 64 == 0:
            stream.synchronize()
    stream.synchronize()
    K = args.steps
    ev_mid = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_end = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(K):
            step(i)
        stop.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    total_ms = start.elapsed_time(stop)
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        b0.record(stream)
        for i in range(K):
            second(i)
        b1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    dom_b2b_ms = b0.elapsed_time(b1) / K
    with torch.cuda.stream(stream):
        for i in range(K):
            first(i)
            ev_mid[i].record(stream)
            second(i)
            ev_end[i].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    dom_ms = [ev_mid[i].elapsed_time(ev_end[i]) for i in range(K)]
    return {"total_ms": total_ms, "dominant_ms": dom_b2b_ms, "dominant_ms_events": dom_ms, "clocks": clocks}


def e2e_int4(args, r, case, signs, scale, ws, S, dev, stream, dec_bytes):
    """Public API from pinned host memory: H2D inputs, write + decode, D2H output, sync.

    The step's host inputs (q, the new tokens' K and V, slot_mapping, seq_lens, block table) sit in
    one pinned staging buffer at 256-byte aligned offsets and go over in one copy (kvq_copy: the
    SMs read the pinned buffer over the chip-to-chip link, so the copy is a kernel node of the
    graph); the API calls take views of the device copy, and the output goes back to pinned memory
    the same way. The step (copy in, write, decode, copy out) is replayed as one CUDA graph through
    kvq.CapturedStep, and the host waits for it every step."""
    names = ("q", "k_new", "v_new", "slots", "lens", "bt")
    srcs = {k: getattr(r, k) for k in names}
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += -(-srcs[k].numel() * srcs[k].element_size() // 256) * 256
    h_buf = torch.empty((total,), dtype=torch.uint8).pin_memory()
    d_buf = torch.empty((total,), dtype=torch.uint8, device=dev)
    d = {}
    for k in names:
        t = srcs[k]
        nbytes = t.numel() * t.element_size()
        h_buf[offs[k]:offs[k] + nbytes].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        d[k] = d_buf[offs[k]:offs[k] + nbytes].view(t.dtype).view(t.shape)
    out_h = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    h2d = total
    d2h = out_h.numel() * out_h.element_size()

    # the public API's prepared calls (the fixed buffers are checked once), replayed as one CUDA
    # graph per step: the host-to-device copy of the staging buffer, the write, the decode and the
    # output's copy back to pinned memory; the host then waits for the step
    writer = kvq.Int4Writer(r.kc, r.vc, r.ks, r.vs, signs)
    decoder = kvq.Int4Decoder(r.kc, r.vc, r.ks, r.vs, d["bt"], d["lens"], signs, scale, case.Hq, num_splits=S,
                              workspace=ws)

    def calls():
        kvq.kvq_copy(d_buf, h_buf, stream=stream)  # pinned host -> device by the SMs: a kernel node
        writer(d["k_new"], d["v_new"], d["slots"], stream=stream)
        decoder(d["q"], r.out, stream=stream)
        kvq.kvq_copy(out_h, r.out, stream=stream)

    captured = kvq.CapturedStep(calls, stream)

    def step():
        captured()
        stream.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    n = max(args.steps, 20)
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    dt = (time.perf_counter() - t0) / n
    return {"seconds_per_step": dt, "bytes": dec_bytes, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def run_tq(args, dist, dev, stream):
    bits = 4 if args.workload.endswith("v4") else 3
    case = workloads.turboquant_fp8(bits)
    B, Hq, Hk, D = case.B, case.Hq, case.Hk, case.D
    sb = workloads.turboquant_slot_bytes(D, bits)
    bt, nb = workloads.paged_layout(case.seq_lens, 10 * dist.rank, num_blocks=None)
    g = torch.Generator(device=dev)
    g.manual_seed(3000 + dist.rank)
    cache = torch.randint(0, 256, (nb, 16, Hk, sb), dtype=torch.uint8, device=dev, generator=g)
    cache[..., :D] &= 0x77  # keep every key code finite (no E4M3 NaN) and moderate
    vdb = -(-D * bits // 8)
    sc = torch.full((nb, 16, Hk), 0.05, dtype=torch.float16, device=dev).view(torch.uint8).view(nb, 16, Hk, 2)
    cache[..., D + vdb:D + vdb + 2] = sc
    cache[..., D + vdb + 2:D + vdb + 4] = 0
    bt = bt.to(dev)
    lens = torch.tensor(case.seq_lens, dtype=torch.int32, device=dev)
    q = torch.randn((B, Hq, D), device=dev, generator=g)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.zeros((kvq.kvq_decode_workspace_bytes(B, Hq, Hk, D, 0),), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D)

    def decode(i):
        kvq.kvq_decode_tq(q, cache, bits, bt, lens, scale, out=out, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        decode(0)
    stream.synchronize()
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd, stream=stream):
        decode(0)
    res = timed_steps(args, dist, stream, lambda i: None, lambda i: gd.replay(), dev.index)
    kvb = sum(case.seq_lens) * Hk * sb
    byt = kvb + sum(-(-L // 16) * 4 for L in case.seq_lens) + B * Hq * D * 8
    cfg = {"workload": args.workload, "B": B, "Hq": Hq, "Hk": Hk, "D": D, "block_size": 16, "seq_len": 4096,
           "slot_bytes": sb, "value_bits": bits, "key": "fp8 e4m3", "num_splits": "heuristic (balanced)",
           "l2": "single %.0f MB cache read per step (> L2)" % (kvb / 1e6), "decode_bytes_per_step": byt}
    return finish(args, dist, res, byt, cfg, None, 2, "decode_tq_v%d" % bits,
                  ["quantized_paged_kv_int4_gb300/csrc/decode_tq.cu",
                   "quantized_paged_kv_int4_gb300/csrc/decode_common.cuh",
                   "quantized_paged_kv_int4_gb300/csrc/kvq_device.cuh"], "f32")


def run_tq_mse(args, dist, dev, stream):
    kb, vb = 3, 4
    case = workloads.turboquant_mse(kb, vb)
    B, Hq, Hk, D = case.B, case.Hq, case.Hk, case.D
    mse, kps, sb = workloads.turboquant_mse_layout(D, kb, vb)
    bt, nb = workloads.paged_layout(case.seq_lens, 10 * dist.rank, num_blocks=None)
    g = torch.Generator(device=dev)
    g.manual_seed(4000 + dist.rank)
    cache = torch.randint(0, 256, (nb, 16, Hk, sb), dtype=torch.uint8, device=dev, generator=g)
    two = lambda x: torch.full((nb, 16, Hk), x, dtype=torch.float16, device=dev).view(torch.uint8).view(nb, 16, Hk, 2)
    cache[..., mse:mse + 2] = two(4.0)                       # key norms
    vdb = -(-D * vb // 8)
    cache[..., kps + vdb:kps + vdb + 2] = two(0.05)          # value scale
    cache[..., kps + vdb + 2:kps + vdb + 4] = 0              # value zero
    bt = bt.to(dev)
    lens = torch.tensor(case.seq_lens, dtype=torch.int32, device=dev)
    q = torch.randn((B, Hq, D), device=dev, generator=g)
    Pi = workloads.random_rotation(D, 1).to(dev)
    cb = workloads.mse_codebook(kb, D).to(dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.zeros((kvq.kvq_decode_tq_mse_workspace_bytes(B, Hq, Hk, D, 0),), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D)

    def decode(i):
        kvq.kvq_decode_tq_mse(q, Pi, cb, cache, kb, kps, vb, bt, lens, scale, out=out, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        decode(0)
    stream.synchronize()
    st, flags = kvq.kvq_device_error(stream)
    assert st == 0, flags
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd, stream=stream):
        decode(0)
    res = timed_steps(args, dist, stream, lambda i: None, lambda i: gd.replay(), dev.index)
    kvb = sum(case.seq_lens) * Hk * sb
    byt = kvb + sum(-(-L // 16) * 4 for L in case.seq_lens) + B * Hq * D * 8 + D * D * 4 + (1 << kb) * 4
    cfg = {"workload": args.workload, "B": B, "Hq": Hq, "Hk": Hk, "D": D, "block_size": 16, "seq_len": 4096,
           "slot_bytes": sb, "key": "MSE %d-bit centroid indices + fp16 norm (key_packed_size %d)" % (kb, kps),
           "value_bits": vb, "num_splits": "heuristic (balanced)",
           "l2": "single %.0f MB cache read per step (> L2)" % (kvb / 1e6), "decode_bytes_per_step": byt}
    return finish(args, dist, res, byt, cfg, None, 3, "decode_tq_mse_k%dv%d" % (kb, vb),
                  ["quantized_paged_kv_int4_gb300/csrc/decode_tq_mse.cu",
                   "quantized_paged_kv_int4_gb300/csrc/decode_common.cuh",
                   "quantized_paged_kv_int4_gb300/csrc/kvq_device.cuh"], "f32")


def run_kpool(args, dist, dev, stream):
    """kpool compress-and-write: 16384 pools of 4 tokens (65536 tokens), pages of 64, four input
    replicas (4 x 50 MB > L2)."""
    n, pool, ps = 16384, 4, 64
    reps = []
    for r in range(4):
        slot_k, score, ape, loc, nb = workloads.kpool_case(n, pool, ps, seed=10 * dist.rank + r)
        reps.append([t.to(dev) for t in (slot_k, score, ape, loc)] +
                    [torch.zeros((nb, ps, 132), dtype=torch.uint8, device=dev)])

    def step(i):
        k, sc, ap, lc, cache = reps[i % 4]
        kvq.kvq_kpool_write(cache, k, sc, ap, lc, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(4):
            step(i)
    stream.synchronize()
    st, flags = kvq.kvq_device_error(stream)
    assert st == 0, flags
    graphs = []
    for i in range(4):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(i)
        graphs.append(g)
    res = timed_steps(args, dist, stream, lambda i: None, lambda i: graphs[i % 4].replay(), dev.index)
    byt = n * pool * 128 * (2 + 4) + pool * 128 * 4 + n * 8 + n * 132
    cfg = {"workload": "kpool_write", "n_pools": n, "pool_size": pool, "page_size": ps, "head_dim": 128,
           "round_scale": True, "l2": "4 rotating input replicas (4 x %.0f MB > 126 MB L2)" % (byt / 1e6),
           "kpool_bytes_per_step": byt}
    return finish(args, dist, res, byt, cfg, None, 1, "kpool_write", ["quantized_paged_kv_int4_gb300/csrc/kpool.cu",
                  "quantized_paged_kv_int4_gb300/csrc/kvq_device.cuh"], "f32")


def run_kpool_update(args, dist, dev, stream):
    """Batched kpool decode update (spec verify): 1024 requests x next_n = 4 tokens, pools of 4 (each
    request completes one pool per step), ring 8, pages of 64."""
    R, nn, pool, ring, ps = 1024, 4, 4, 8, 64
    g = torch.Generator().manual_seed(50 + dist.rank)
    key = torch.randn((R, nn, 128), generator=g).to(torch.bfloat16).to(dev)
    score = (torch.randn((R, nn, 128), generator=g) * 2).to(torch.bfloat16).to(dev)
    ape = (torch.randn((pool, 128), generator=g) * 0.5).to(dev)
    tail = (torch.randn((R, 2, ring, 128), generator=g)).to(torch.bfloat16).to(dev)
    nb = R // ps + 4
    cache = torch.zeros((nb, ps, 132), dtype=torch.uint8, device=dev)
    pos = (torch.arange(nn, dtype=torch.int32)[None, :] + 100).repeat(R, 1)          # positions 100..103
    ts = (torch.arange(R, dtype=torch.int32)[:, None] * ring + pos % ring).to(torch.int32)
    loc = torch.where(pos % pool == pool - 1, torch.randperm(nb * ps, generator=g)[:R, None].to(torch.int32),
                      torch.full_like(pos, -1))
    pos, ts, loc = pos.to(dev), ts.to(dev), loc.to(dev)

    def step(i):
        kvq.kvq_kpool_decode_update(cache, tail, ts, key, score, ape, loc, pos, pool, stream=stream)

    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    st, flags = kvq.kvq_device_error(stream)
    assert st == 0, flags
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        step(0)
    res = timed_steps(args, dist, stream, lambda i: None, lambda i: gr.replay(), dev.index)
    byt = R * nn * 128 * 2 * 2 + R * (pool - 1) * 128 * 2 * 2 + R * nn * 128 * 2 * 2 + R * 132 + 3 * R * nn * 4
    cfg = {"workload": "kpool_decode_update", "requests": R, "next_n": nn, "pool_size": pool, "ring": ring,
           "page_size": ps, "l2": "inputs %.1f MB (L2-resident; a launch-latency-bound step)" % (byt / 1e6),
           "kpool_update_bytes_per_step": byt}
    return finish(args, dist, res, byt, cfg, None, 1, "kpool_decode_update",
                  ["quantized_paged_kv_int4_gb300/csrc/kpool.cu", "quantized_paged_kv_int4_gb300/csrc/kvq_device.cuh"],
                  "f32")


def run_write_fwht(args, dist, dev, stream):
    nrep = 4
    reps = []
    signs = workloads.rht_signs(128).to(dev)
    for r in range(nrep):
        k, v, slots, nb = workloads.write_case(seed=10 * dist.rank + r)
        kc = torch.zeros((nb, 16, 8, 64), dtype=torch.uint8, device=dev)
        reps.append(dict(k=k.to(dev), v=v.to(dev), slots=slots.to(dev), kc=kc, vc=torch.zeros_like(kc),
                         ks=torch.zeros((nb, 16, 8), dtype=torch.float32, device=dev),
                         vs=torch.zeros((nb, 16, 8), dtype=torch.float32, device=dev),
                         x=workloads.fwht_rows(65536, seed=r).to(dev),
                         y=torch.empty((65536, 128), dtype=torch.float8_e4m3fn, device=dev),
                         s=torch.empty((65536, 1), dtype=torch.float32, device=dev)))
    live = int((reps[0]["slots"] >= 0).sum())

    def write(i):
        r = reps[i % nrep]
        kvq.kvq_write_int4(r["k"], r["v"], r["kc"], r["vc"], r["ks"], r["vs"], r["slots"], signs, stream=stream)

    def fwht(i):
        r = reps[i % nrep]
        kvq.kvq_fwht128(r["x"], r["y"], r["s"], stream=stream)

    with torch.cuda.stream(stream):
        for i in range(nrep):
            write(i)
            fwht(i)
    stream.synchronize()
    gw, gf = [], []
    for i in range(nrep):
        a, b = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(a, stream=stream):
            write(i)
        with torch.cuda.graph(b, stream=stream):
            fwht(i)
        gw.append(a)
        gf.append(b)
    # the dominant call here is the write: time it between the events
    res = timed_steps(args, dist, stream, lambda i: gf[i % nrep].replay(), lambda i: gw[i % nrep].replay(), dev.index)
    wr = live * 8 * (2 * 128 * 2 + 2 * (64 + 4)) + 16384 * 8
    fw = 65536 * (256 + 128 + 4)
    cfg = {"workload": "write_fwht", "write": "16384 tokens x Hk 8 x D 128 bf16, 5%% slot_mapping = -1 (%d live)" % live,
           "fwht": "65536 x 128 bf16 -> e4m3 + fp32 scale", "l2": "4 rotating input replicas (> L2)",
           "write_bytes_per_step": wr, "fwht_bytes_per_step": fw}
    return finish(args, dist, res, wr + fw, cfg, None, 2, "write_int4", ["quantized_paged_kv_int4_gb300/csrc/write_int4.cu",
                  "quantized_paged_kv_int4_gb300/csrc/kvq_device.cuh"], "f32", dom_bytes=wr)


def finish(args, dist, res, step_bytes, cfg, e2e, kernels_per_step, dom_tag, dom_sources, dtype, dom_bytes=None):
    K = args.steps
    ms = dist.max(res["total_ms"] / K)
    total_bytes = dist.sum(step_bytes)
    value = total_bytes / (ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    dom_ms = dist.max(res["dominant_ms"])
    dom_ev_ms = statistics.mean(res["dominant_ms_events"])
    dom_b = step_bytes if dom_bytes is None else dom_bytes
    achieved = dom_b / (dom_ms * 1e-3) / 1e9
    traffic = ncu_traffic(dom_tag, dom_sources)
    data = ("synthetic: seeded queries; the paged INT4 cache written by kvq_write_int4 from K ~ N(0,1) "
            "(outlier channels x10) and V ~ N(0,1)" if dom_tag.startswith("decode_int4") else
            "synthetic (seeded random caches and queries of the workload's shapes)")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "us_per_step": round(ms * 1e3, 2),
        "pct_hbm_peak": round(100.0 * (step_bytes / (ms * 1e-3) / 1e9) / peak, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": data,
        "config": cfg, "clocks": res["clocks"], "gpu_launches": kernels_per_step * K,
        "roofline": {"bound": "hbm", "kernel": dom_tag, "achieved": round(achieved, 2), "peak": peak,
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_src if peak_src == "measured"
                     else "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": dom_b,
                     "avg_launch_us": round(dom_ms * 1e3, 3),
                     "avg_launch_us_timing": "K calls back to back between one event pair (inputs rotate over "
                                             "replicas larger than L2)",
                     "avg_launch_us_with_events": round(dom_ev_ms * 1e3, 3),
                     "note": ("launch = the whole library call (q rotation, split-KV kernel, LSE merge kernel)"
                              if dom_tag.startswith("decode_tq_mse") else
                              "launch = the whole library call (q rotation kernel for plain single-token calls, "
                              "split-KV kernel, LSE merge kernel)")
                     if dom_tag.startswith("decode") else "launch = one %s kernel" % dom_tag},
    }
    if e2e is not None:
        e_s = dist.max(e2e["seconds_per_step"])
        line["e2e"] = {"value": round(total_bytes / e_s / 1e9, 2), "unit": "GB/s", "us_per_step": round(e_s * 1e6, 2),
                       "h2d_bytes_per_step": e2e["h2d_bytes_per_step"], "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and args.workload == "llama3_8b_int4":
        line["cpu_baseline"] = cpu_baseline(budget_s=20.0)
    return line


# ----------------------------------------------------------------------------------------------
# CPU oracle (test infrastructure): the cpu_baseline leg and the --impl reference arm
# ----------------------------------------------------------------------------------------------
def _oracle_sample(seqs, seed=0):
    from oracle import int4_cache
    case = workloads.llama8b_int4()
    lens = [case.seq_lens[b] for b in seqs]
    bt, nb = workloads.paged_layout(lens, seed)
    kb, vb, kw, vw = workloads.random_int4_pages(nb, case.Hk, case.D, seed)
    q = workloads.to_numpy_f32(workloads.query(case)[seqs])
    signs = workloads.rht_signs(case.D).numpy()
    args = (q, kb.numpy(), vb.numpy(), kw.numpy().view(np.uint32), vw.numpy().view(np.uint32), bt.numpy(),
            np.asarray(lens), signs, 1.0 / math.sqrt(case.D))
    byts, _ = int4_decode_bytes(lens, case.Hq, case.Hk, case.D)
    return int4_cache.decode_int4, args, byts


def _oracle_worker(seqs, barrier):
    """One process of the all-cores leg: prepare its sequences' inputs, wait for every worker,
    then run the oracle on them; returns (start, end, bytes)."""
    jobs = [_oracle_sample([b]) for b in seqs]
    barrier.wait()
    t0 = time.time()
    byts = 0
    for fn, a, nbytes in jobs:
        fn(*a)
        byts += nbytes
    return t0, time.time(), byts


def cpu_baseline_parallel(n_workers=None):
    """The oracle on all host cores: the 32 sequences of one step dealt round-robin to one
    spawned process per core (the pool starts after the GPU work, so spawn, never fork), timed from
    the common start to the last worker's end."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    n = n_workers or os.cpu_count() or 1
    n = max(1, min(n, 32))
    ctx = mp.get_context("spawn")
    env = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env:
        os.environ[k] = "1"  # one thread per worker process
    try:
        with ctx.Manager() as mgr:
            barrier = mgr.Barrier(n)
            with ProcessPoolExecutor(max_workers=n, mp_context=ctx) as ex:
                futs = [ex.submit(_oracle_worker, list(range(w, 32, n)), barrier) for w in range(n)]
                res = [f.result() for f in futs]
    finally:
        for k, v in env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    t0 = min(r[0] for r in res)
    t1 = max(r[1] for r in res)
    byts = sum(r[2] for r in res)
    return {"value": round(byts / (t1 - t0) / 1e9, 5), "unit": "GB/s", "cores": n, "kind": "oracle",
            "seconds": round(t1 - t0, 2),
            "sample": "all 32 sequences of one step, one spawned process per core (float64 numpy oracle)"}


def cpu_baseline(budget_s=20.0):
    """The oracle as it stands, single-threaded numpy, on consecutive sequences of the workload
    until ~budget_s of CPU time (or the whole batch); plus the same oracle on all host cores."""
    done, byts, spent = [], 0, 0.0
    for b in range(32):
        fn, a, nbytes = _oracle_sample([b])
        t0 = time.perf_counter()
        fn(*a)
        spent += time.perf_counter() - t0
        done.append(b)
        byts += nbytes
        if spent >= budget_s:
            break
    line = {"value": round(byts / spent / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(spent, 2),
            "sample": "%d of the 32 sequences of one step (float64 numpy oracle, one thread)" % len(done)}
    try:
        line["all_cores"] = cpu_baseline_parallel()
        line["nproc"] = os.cpu_count()
    except Exception as e:  # the single-thread figure stands on its own
        line["all_cores"] = {"unavailable": "%s: %s" % (type(e).__name__, e)}
    return line


def run_reference(args, dist):
    if dist.rank != 0:
        return None
    seqs = [0, 1]
    fn, a, nbytes = _oracle_sample(seqs)
    for _ in range(args.warmup):
        fn(*a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn(*a)
    dt = (time.perf_counter() - t0) / args.steps
    v = round(nbytes / dt / 1e9, 5)
    case = workloads.llama8b_int4()
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": "llama3_8b_int4", "B": case.B, "Hq": case.Hq,
                                            "Hk": case.Hk, "D": case.D, "sample_sequences": seqs},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "sequences 0 and 1 of the workload per step (float64 numpy oracle)"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            line = run_reference(args, dist)
        else:
            if not torch.cuda.is_available():
                raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
            line = run_kvq(args, dist)
        if line is not None and dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
