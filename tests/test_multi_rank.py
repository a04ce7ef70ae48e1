"""The bench's multi-rank host path on CPU ranks (gloo, world size 2): replicas share nothing but
the max over ranks of the timed region, and only rank 0 prints the reference arm's line."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.slowest_rank_seconds(times[rank], world)
        q.put((rank, t, bench.job_value(world, 1e9, t)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_job_value_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.5, 0.8]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [0.8, 0.8]                  # every rank sees the slowest
    assert all(abs(g[2] - 2 * 1e9 / 0.8 / 1e9) < 1e-12 for g in got)


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_seconds(0.25, 1) == 0.25


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                          "--steps", "1", "--warmup", "3"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == "", out.stderr[-500:]
