"""The benchmark's multi-rank host logic on the CPU (gloo, world size 2).

Each GPU runs its own replica of the workload (the GEMV needs no exchange between
GPUs); the reported value is all ranks' bytes over the slowest rank's step time.
These tests run the aggregation over a real two-process gloo group, and check that
the CPU reference arm prints only on rank 0.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]          # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, dist)
        value = bench.whole_job_gbs(world, 10**9, slowest)
        dist.barrier()
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_whole_job_over_slowest_rank():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks agree on the slowest time and on the whole-job throughput
    assert [m for _, m, _ in got] == [5.0, 5.0]
    for _, _, v in got:
        assert abs(v - 2 * 1e9 / 5e-3 / 1e9) < 1e-9   # 2 ranks x 1 GB in 5 ms = 400 GB/s


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.max_over_ranks(7.5, None) == 7.5
    assert bench.whole_job_gbs(1, 268517376, 45.0e-3) == pytest.approx(5967.05, rel=1e-4)


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "0"], env=env, cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_only_on_rank_zero():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
    r = _run_reference({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
