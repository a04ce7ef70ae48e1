"""One decode step from host memory through hw_decode_step_host (needs a GPU).

Inputs go up packed ([K][V][Q] of every layer, page-locked) and outputs come back to host
memory; in between the library runs the same append, attention and step end as the device
calls.  Every step's host output is compared with the fp64 oracle (1e-2 max-abs, the parity
tolerance), with commits between steps, on both attention kernels, one and several layers,
bf16 and fp32 output, synchronous and enqueue-only calls; then the tables and stored pools.
Refused calls enqueue nothing and leave the context as it was.
"""
import dataclasses

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


def run_host_steps(w, steps, out_dtype="bf16", bernoulli=None, sync_every=1,
                   small_scratch=False):
    """``steps`` decode steps through hw_decode_step_host; with sync_every > 1 only every
    sync_every-th call synchronises (the others only enqueue, each with its own buffers).
    small_scratch: the cache starts with a device scratch too small for a step, which the
    first call must refuse before enqueuing anything and the wrapper then grows."""
    import torch

    import gpu_cases as G
    from oracle import attention as A
    from oracle import run as orun
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    r = WorkloadRunner(w)
    if small_scratch:
        r.cache._step_scratch = torch.empty(256, dtype=torch.uint8, device="cuda")
    P, W, Hq, D, L = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim, w.num_layers
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    ins = [r.packed_inputs(s) for s in range(steps)]
    outs = [torch.full((L, P, W, Hq, D), float("nan"), dtype=dt).pin_memory()
            for _ in range(steps)]
    masks = [wl.finished_mask(w, s, bernoulli) for s in range(steps)]
    for s in range(steps):
        sync = (s + 1) % sync_every == 0 or s + 1 == steps
        r.cache.decode_step_host(r.n_step, ins[s], outs[s], masks[s], out_dtype, sync=sync)
    torch.cuda.synchronize()
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    c = orun.prefill(w)
    worst = 0.0
    for s in range(steps):
        orun.append_step(c, w, s)
        got = outs[s].float().numpy()
        for layer in range(L):
            ref, _ = A.method(c, layer, orun.query(w, layer, s))
            err = float(np.abs(got[layer] - ref).max())
            worst = max(worst, err)
            assert err <= G.TOL, (s, layer, err)
        c.step_end(masks[s])
    G.dev_tables_equal(r, c)
    for layer in range(L):
        G.check_pools(r, c, layer, 64)
    r.cache.close()
    return worst


def test_host_step_tensor_cores_with_commits():
    """8 workers, 64 rows per KV head (tensor-core kernel), a 9000-token common block, random
    commits between steps."""
    w = dataclasses.replace(wl.c4(), common_len=(9000,), steps=8)
    run_host_steps(w, 6, bernoulli=0.3)


def test_host_step_cuda_core_kernel():
    w = dataclasses.replace(wl.tiny(), steps=5)
    run_host_steps(w, 4, bernoulli=0.5)


def test_host_step_scratch_grown_after_the_refusal():
    w = dataclasses.replace(wl.tiny(), steps=4)
    run_host_steps(w, 3, small_scratch=True)


def test_host_step_layers_fp32_enqueue_only():
    """Three layers, fp32 output; only every third call synchronises."""
    w = dataclasses.replace(wl.c3(), num_layers=3, common_len=(3000,), steps=8)
    run_host_steps(w, 6, out_dtype="f32", sync_every=3)


def test_host_step_several_problems_step_wise():
    w = dataclasses.replace(wl.c5(), num_problems=3, common_len=(700, 2100, 1300),
                            worker_len=((9, 0, 130, 20), (3, 5, 0, 1), (256, 255, 1, 0)), steps=5,
                            layout="step_wise", commit_steps=(1, 3))
    run_host_steps(w, 4)


def test_host_step_refusals_enqueue_nothing():
    import torch
    from shared_kv_concurrent_gb300 import HogwildError, binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    w = dataclasses.replace(wl.tiny(), steps=3)
    r = WorkloadRunner(w)
    ctx = r.cache.ctx
    inp = r.packed_inputs(0)
    out = torch.zeros(w.num_layers * w.num_problems * w.num_workers * w.num_q_heads * w.head_dim,
                      dtype=torch.bfloat16).pin_memory()
    need = binding.hw_step_scratch_size(ctx, r.n_step, binding.HW_OUT_BF16)
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    before = r.cache.tables()
    cases = [
        (dict(in_bytes=inp.numel() - 2), binding.HW_ERR_INVALID_ARG),
        (dict(scratch_bytes=need - 1), binding.HW_ERR_CAPACITY),
        (dict(out_dtype=7), binding.HW_ERR_INVALID_ARG),
        (dict(scratch=scratch.data_ptr() + 16, scratch_bytes=need - 16), binding.HW_ERR_INVALID_ARG),
    ]
    for over, status in cases:
        kw = dict(in_bytes=inp.numel(), scratch=scratch.data_ptr(), scratch_bytes=need,
                  out_dtype=binding.HW_OUT_BF16)
        kw.update(over)
        with pytest.raises(HogwildError) as e:
            binding.hw_decode_step_host(ctx, r.n_step, inp.data_ptr(), kw["in_bytes"],
                                        out.data_ptr(), kw["out_dtype"], None, kw["scratch"],
                                        kw["scratch_bytes"])
        assert e.value.status == status
    assert r.cache.tables() == before
    # a step already open
    k, v, _ = r.step_inputs(0)
    r.cache.append_kv(0, r.n_step, k[0], v[0])
    with pytest.raises(HogwildError) as e:
        binding.hw_decode_step_host(ctx, r.n_step, inp.data_ptr(), inp.numel(), out.data_ptr(),
                                    binding.HW_OUT_BF16, None, scratch.data_ptr(), need)
    assert e.value.status == binding.HW_ERR_INVALID_ARG
    r.cache.step_end()
    torch.cuda.synchronize()
    r.cache.close()
