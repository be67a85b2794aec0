"""bench.py's multi-rank logic on two gloo ranks (CPU): the max-over-ranks time, the whole-job
byte sum, the line that rank 0 prints, and the reference arm's rank-0-only rule. No GPU."""

import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()
    try:
        out = {"max": d.max(rank + 1.0), "sum": d.sum(10.0 * (rank + 1))}
        # rank r takes (r + 1) ms per step for (r + 1) GB: the job moved 3 GB per step in the
        # slowest rank's 2 ms
        args = types.SimpleNamespace(steps=4, warmup=3, workload="write_fwht", no_cpu_baseline=True)
        res = {"total_ms": 4.0 * (rank + 1), "dominant_ms": 0.5 * (rank + 1), "dominant_ms_events": [0.6, 0.6],
               "clocks": {"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": []}}
        line = bench.finish(args, d, res, 1e9 * (rank + 1), {"workload": "test"}, None, 2, "write_int4",
                            [], "f32")
        out["line"] = line
        # reference arm: only rank 0 works (a stand-in oracle sample keeps this fast)
        bench._oracle_sample = lambda seqs: (lambda: None, (), 1000)
        ref = bench.run_reference(types.SimpleNamespace(steps=2, warmup=1), d)
        out["ref"] = None if ref is None else ref["impl"]
        d.barrier()
    finally:
        d.close()
    q.put((rank, out))


@pytest.mark.timeout(120)
def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for r in (0, 1):
        assert got[r]["max"] == 2.0 and got[r]["sum"] == 30.0
        line = got[r]["line"]
        assert line["n_gpus"] == 2 and line["steps"] == 4 and line["warmup"] == 3
        assert line["ms_per_step"] == pytest.approx(2.0)            # max over ranks
        assert line["value"] == pytest.approx(3e9 / 2e-3 / 1e9)  # whole-job bytes / slowest time
        assert line["gpu_launches"] == 8 and line["scaling"] == "weak"
        # the dominant call: back-to-back average, max over ranks; the per-call-event figure beside it
        assert line["roofline"]["avg_launch_us"] == pytest.approx(1000.0)
        assert line["roofline"]["avg_launch_us_with_events"] == pytest.approx(600.0)
    assert got[0]["ref"] == "reference" and got[1]["ref"] is None
