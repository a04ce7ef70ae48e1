"""Parity of the exact launch sequence the benchmark times (needs a GPU).

bench.py enqueues many decode steps back to back on one stream with no host synchronisation:
each step is hw_append_kv, hw_concurrent_attention and hw_step_end on one of R independent
caches in turn, all queued behind a device-side delay so that the GPU runs them as one chain.
Consecutive kernels then overlap (programmatic dependent launches): the next step's attention
kernel sets up and loads its first K/V tile while the previous step still runs, and the plans
go up on the library's copy stream without a stream wait.  None of that happens when a test
synchronises after every call, so these tests drive the same pattern -- every step with its
own output buffers, inputs kept alive -- and compare every step against the fp64 oracle only
after one final synchronisation: outputs (1e-2 max-abs), lse, tables and stored pools -- on
both attention kernels (tensor cores from 16 query rows per KV head, CUDA cores below).
"""
import numpy as np
import pytest

import workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from shared_kv_concurrent_gb300.build import build
    build()


def run_chained(w, caches, steps_per_cache, out_dtype="bf16", pool_sample=64):
    """``caches`` independent caches of workload ``w``, ``steps_per_cache`` decode steps each,
    interleaved (step i goes to cache i mod R) and enqueued without a host synchronisation."""
    import time

    import torch

    import gpu_cases as G
    from oracle import attention as A
    from oracle import run as orun
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    R = caches
    runners = [WorkloadRunner(w) for _ in range(R)]
    P, W, Hq, D, L = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim, w.num_layers
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    seq = [(i % R, i // R) for i in range(R * steps_per_cache)]
    # inputs of every step resident on the device before the chain starts (as in the bench)
    inputs = {(c, st): runners[c].step_inputs(st) for c, st in seq}
    outs = {k: [torch.full((P, W, Hq, D), float("nan"), dtype=dt, device="cuda")
                for _ in range(L)] for k in seq}
    lses = {k: [torch.full((P, W, Hq), float("nan"), dtype=torch.float32, device="cuda")
                for _ in range(L)] for k in seq}
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    # a bounded device-side delay, so that the host has queued every step before the GPU starts
    t0 = time.perf_counter()
    torch.cuda._sleep(int(0.05 * 2.07e9))
    for c, st in seq:
        runners[c].append(inputs[(c, st)], stream=stream)
        runners[c].attend(inputs[(c, st)], outs[(c, st)], lses[(c, st)], out_dtype,
                          stream=stream)
        runners[c].end(st, stream=stream)
    host_s = time.perf_counter() - t0
    torch.cuda.synchronize()
    for r in runners:
        st_, info = r.cache.check_device_errors()
        assert st_ == binding.HW_OK, info
    # the oracle, one cache at a time, the same steps in the same order
    worst = 0.0
    for c in range(R):
        oc = orun.prefill(w)
        for st in range(steps_per_cache):
            orun.append_step(oc, w, st)
            for layer in range(L):
                ref, ref_lse = A.method(oc, layer, orun.query(w, layer, st))
                got = outs[(c, st)][layer].float().cpu().numpy()
                err = float(np.abs(got - ref).max())
                worst = max(worst, err)
                assert err <= G.TOL, (c, st, layer, err)
                gl = lses[(c, st)][layer].cpu().numpy()
                fin = np.isfinite(ref_lse)
                assert np.array_equal(np.isfinite(gl), fin)
                assert np.abs(gl[fin] - ref_lse[fin]).max(initial=0.0) <= G.TOL
            oc.step_end(wl.finished_mask(w, st))
        G.dev_tables_equal(runners[c], oc)
        for layer in range(L):
            G.check_pools(runners[c], oc, layer, pool_sample)
        runners[c].cache.close()
    return worst, host_s


def test_chained_scaled_w8_three_caches():
    """8 workers, 64 query rows per KV head (tensor-core kernel), a 9000-token common block and
    the benchmark's own worker blocks; three caches, eight steps each, interleaved."""
    import dataclasses
    w = dataclasses.replace(wl.c4(), common_len=(9000,), steps=10)
    worst, _ = run_chained(w, caches=3, steps_per_cache=8)
    assert worst <= 1e-2


def test_chained_full_size_w8_common32768():
    """The benchmark workload itself, two caches, five steps each."""
    import dataclasses
    w = dataclasses.replace(wl.c4(), steps=6)
    run_chained(w, caches=2, steps_per_cache=5, pool_sample=32)


def test_chained_batch_of_problems_with_commits():
    """A slice of the 16-problem workload with every worker committing after steps 2 and 5, so
    that views, rotations and pieces change inside the chain; two caches, eight steps each."""
    import dataclasses
    w = dataclasses.replace(wl.c5(), num_problems=4, common_len=(1500, 4100, 700, 2600),
                            worker_len=((0, 300, 17, 256), (5, 0, 0, 129), (511, 1, 64, 200),
                                        (40, 40, 0, 90)), steps=9, commit_steps=(2, 5))
    run_chained(w, caches=2, steps_per_cache=8)


def test_chained_multi_layer_fp32_output():
    """Three layers sharing one plan per step (the 64-layer workload's shape), fp32 output."""
    import dataclasses
    w = dataclasses.replace(wl.c3(), num_layers=3, common_len=(3000,), steps=6)
    run_chained(w, caches=2, steps_per_cache=5, out_dtype="f32")


def test_chained_cuda_core_w2_contiguous():
    """The 2-worker contiguous workload: 10 query rows per KV head, the CUDA-core kernel, whose
    set-up (plan check, unit record, first tile, first rotation factors) runs before its grid
    wait and writes the step's tokens itself; three caches, six steps each."""
    import dataclasses
    w = dataclasses.replace(wl.c2(), steps=7)
    run_chained(w, caches=3, steps_per_cache=6)


def test_chained_cuda_core_head_dim_64_with_commits():
    """8 rows at head dim 64 (CUDA-core kernel) with both workers committing after steps 1 and
    3; two caches, six steps each."""
    import dataclasses
    w = dataclasses.replace(wl.tiny(), steps=7, commit_steps=(1, 3))
    run_chained(w, caches=2, steps_per_cache=6)
