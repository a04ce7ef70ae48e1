"""Multi-rank host paths on CPU ranks (gloo, world size 2).

The bench's replicas share nothing but the max over ranks of the timed region, and only rank 0
prints the reference arm's line.  The sequence split's exchange (shared_kv_concurrent_gb300.
seqsplit) gathers every rank's (out, lse) part in rank order; here each rank computes its part
with the oracle (the library's kernels need a GPU), and the gathered parts, merged, must give
the attention over the whole view."""
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


def _split_rank(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle.attention as A
    import oracle_pins as pins
    from shared_kv_concurrent_gb300 import seqsplit
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        worst = 0.0
        for c, qq in pins.random_session(5, 64, 3, steps=3):   # the same cache on every rank
            totals = [A.entry_spans(c, p)[1] for p in range(c.P)]
            ranges = seqsplit.split_entries(totals, world)[rank]
            out, lse = A.method_range(c, 0, qq, ranges)
            po, pl = seqsplit.gather_parts(torch.from_numpy(out), torch.from_numpy(lse))
            assert torch.equal(po[rank], torch.from_numpy(out))          # rank order
            mo, ml = A.merge_parts(po.numpy(), pl.numpy())
            ro, rl = A.method(c, 0, qq)
            worst = max(worst, float(np.abs(mo - ro).max()))
            fin = np.isfinite(rl)
            assert np.array_equal(np.isfinite(ml), fin)
            assert np.abs(ml[fin] - rl[fin]).max() <= 1e-10
        q.put((rank, worst))
    finally:
        dist.destroy_process_group()


def test_sequence_split_exchange_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1] and all(g[1] <= 1e-10 for g in got), got


def test_split_entries_partitions_every_problem():
    sys.path.insert(0, ROOT)
    from shared_kv_concurrent_gb300.seqsplit import split_entries
    for totals, world in (([10, 7, 0], 3), ([1], 4), ([37726], 2), ([5, 5], 1)):
        r = split_entries(totals, world)
        assert r.shape == (world, len(totals), 2)
        for p, n in enumerate(totals):
            assert r[0, p, 0] == 0 and r[-1, p, 1] == n
            assert all(r[k, p, 1] == r[k + 1, p, 0] for k in range(world - 1))
            sizes = r[:, p, 1] - r[:, p, 0]
            assert sizes.min() >= 0 and sizes.max() - sizes.min() <= 1
