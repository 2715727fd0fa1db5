"""The multi-process path of the benchmark on CPU: two gloo ranks (no GPU).

Replicas only: every rank runs the same workload on its own data, the
timing takes the slowest rank, and the whole-job rate counts every rank's
units.  The reference arm under a 2-rank launcher prints one line from
rank 0 and exits cleanly on rank 1.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slower one
        slowest = bench.max_over_ranks(local_ms, world, "cpu")
        rate = bench.whole_job_rate(1000, slowest, 4, world)
        q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_timing_and_whole_job_rate_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, rate in got:
        assert slowest == 15.0                            # every rank sees the max
        assert rate == pytest.approx(2 * 1000 / (15.0 / 1e3 / 4))


def test_single_rank_passes_values_through():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(10, 2.0, 1, 1) == pytest.approx(5000.0)


def test_replicas_draw_different_data_per_rank():
    from paged_kv_cache_307_gb300 import workloads as W
    s = W.SPECS["c2"]
    a = W.decode_case("c2", small=True, seed=s.seed + 1000 * 0, nan_fill=False)
    b = W.decode_case("c2", small=True, seed=s.seed + 1000 * 1, nan_fill=False)
    assert not torch.equal(a.q, b.q)


def test_reference_arm_under_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=%d" % port, os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    # the line carries the same metric and workload as the CUDA arm, and the
    # oracle's own timing as both its cpu_baseline and its end-to-end figure
    assert d["metric"].startswith("paged decode attention HBM GB/s") and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 0
    assert d["config"]["workload"].startswith("c2")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
