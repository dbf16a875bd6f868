"""Host logic of bench.py for N > 1 ranks, run as gloo processes on the CPU.

Rows are independent, so N GPUs run N replicas of the workload (weak
scaling) with no data-path collective; the only cross-rank steps are the
barrier around the timed region and the max over ranks of the step time.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, local = bench.dist_env()
    bench.init_dist(w, r)
    slowest = bench.max_over_ranks(times[r], w)
    q.put((r, local, torch.distributed.get_backend(), slowest, bench.aggregate_gbs(3e9, w, slowest)))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_dist_env_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(2.5, 1) == 2.5
    # one rank moving 6.4e9 bytes in 1 ms is 6400 GB/s; two replicas in the same time, twice that
    assert bench.aggregate_gbs(6.4e9, 1, 1.0) == pytest.approx(6400.0)
    assert bench.aggregate_gbs(6.4e9, 2, 1.0) == pytest.approx(12800.0)


def test_max_over_ranks_world2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [1.5, 4.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [g[0] for g in got] == [0, 1]
    assert [g[1] for g in got] == [0, 1]  # LOCAL_RANK picks the device of each rank
    assert all(g[2] == "gloo" for g in got)
    # every rank reports the slowest rank's time, and the job-wide rate over it
    assert [g[3] for g in got] == [4.0, 4.0]
    assert all(g[4] == pytest.approx(3e9 * 2 / 4.0e6) for g in got)
    assert all(p.exitcode == 0 for p in procs)


def test_reference_arm_world2_prints_one_line():
    """Under torchrun with two ranks, rank 0 alone times the oracle and prints
    one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--workload",
           "tiny_causal_f32", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_causal_f32"
