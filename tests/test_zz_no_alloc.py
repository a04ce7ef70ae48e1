"""The allocation-free attention entry point (needs a GPU).

hw_concurrent_attention_noalloc serves callers that cannot allocate device memory when they
call it; its plan and partial results live in a fixed 16 MiB device array inside the library.
It must give the same result as hw_concurrent_attention -- checked on two calls in a row, so
that contents left in the shared array by the first call cannot leak into the second -- and
must refuse a problem whose partial results cannot fit in the array.  This file is collected
last so that a failure here never hides another test.
"""
import pytest

import workload as wl

pytestmark = pytest.mark.gpu

TOL = 1e-2          # the tolerance of the parity tests (max-abs, bf16 inputs, fp32 accumulation)


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from shared_kv_concurrent_gb300.build import build
    build()


def _small_w8():
    import dataclasses
    return dataclasses.replace(wl.c4(), common_len=(3001,),
                               worker_len=((0, 1, 127, 128, 129, 255, 257, 600),), steps=3)


def test_matches_regular_entry_point_on_two_calls_in_a_row():
    import torch
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    w = _small_w8()
    r = WorkloadRunner(w)
    ctx = r.cache.ctx
    shape = (w.num_problems, w.num_workers, w.num_q_heads, w.head_dim)
    for step in range(2):
        inputs = r.step_inputs(step)
        r.append(inputs)
        q = inputs[2][0]
        ref = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        ref_lse = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        binding.hw_concurrent_attention(ctx, 0, q, ref, binding.HW_OUT_F32, ref_lse)
        got = torch.full_like(ref, float("nan"))
        got_lse = torch.full_like(ref_lse, float("nan"))
        binding.hw_concurrent_attention_noalloc(ctx, 0, q, got, binding.HW_OUT_F32, got_lse)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all() and torch.isfinite(got_lse).all()
        assert (got - ref).abs().max().item() <= TOL
        assert (got_lse - ref_lse).abs().max().item() <= TOL
        r.end(step)
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    r.cache.close()


def test_refuses_partials_beyond_the_array():
    import torch
    from shared_kv_concurrent_gb300 import HogwildCache, HogwildError, binding, config_for
    # 40 problems x 8 KV heads x 128 rows x 132 floats x 4 B = 21.6 MB of partials > 16 MiB.
    cfg = config_for(num_problems=40, num_workers=16, num_layers=1, num_q_heads=64,
                     num_kv_heads=8, head_dim=128, page_size=128, num_pages=4,
                     max_position=1024, rope_theta=1e6)
    c = HogwildCache(cfg)
    q = torch.zeros(40, 16, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(HogwildError) as e:
        binding.hw_concurrent_attention_noalloc(c.ctx, 0, q, out, binding.HW_OUT_F32)
    assert e.value.status == binding.HW_ERR_CAPACITY
    c.close()


def test_first_in_its_step_then_the_regular_call():
    """The allocation-free call made first in a step, right after the append, so that it writes
    the layer's recorded append itself; a second cache fed the same inputs gives the reference
    through the regular call.  The regular call made afterwards in the same step still
    matches."""
    import torch
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    w = _small_w8()
    r1, r2 = WorkloadRunner(w), WorkloadRunner(w)
    shape = (w.num_problems, w.num_workers, w.num_q_heads, w.head_dim)
    for step in range(2):
        inputs = r1.step_inputs(step)
        r1.append(inputs)
        r2.append(inputs)
        q = inputs[2][0]
        got = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        got_lse = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        binding.hw_concurrent_attention_noalloc(r1.cache.ctx, 0, q, got, binding.HW_OUT_F32,
                                                got_lse)
        ref = torch.full_like(got, float("nan"))
        ref_lse = torch.full_like(got_lse, float("nan"))
        binding.hw_concurrent_attention(r2.cache.ctx, 0, q, ref, binding.HW_OUT_F32, ref_lse)
        after = torch.full_like(got, float("nan"))
        binding.hw_concurrent_attention(r1.cache.ctx, 0, q, after, binding.HW_OUT_F32)
        torch.cuda.synchronize()
        assert (got - ref).abs().max().item() <= TOL
        assert (got_lse - ref_lse).abs().max().item() <= TOL
        assert (after - ref).abs().max().item() <= TOL
        r1.end(step)
        r2.end(step)
    for r in (r1, r2):
        st, info = r.cache.check_device_errors()
        assert st == binding.HW_OK, info
        r.cache.close()


# The refused call enqueues nothing, so the captured graph is empty and torch says so.
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_refused_on_a_capturing_stream():
    """A stream that is capturing a CUDA graph is refused before anything is enqueued; the
    same call on the same stream after the capture works."""
    import torch
    from shared_kv_concurrent_gb300 import HogwildError, binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    w = _small_w8()
    r = WorkloadRunner(w)
    inputs = r.step_inputs(0)
    r.append(inputs)
    q = inputs[2][0]
    shape = (w.num_problems, w.num_workers, w.num_q_heads, w.head_dim)
    out = torch.zeros(shape, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    status = None
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        try:
            binding.hw_concurrent_attention_noalloc(r.cache.ctx, 0, q, out, binding.HW_OUT_F32,
                                                    None, s)
        except HogwildError as e:
            status = e.status
    assert status == binding.HW_ERR_UNSUPPORTED
    binding.hw_concurrent_attention_noalloc(r.cache.ctx, 0, q, out, binding.HW_OUT_F32, None, s)
    s.synchronize()
    assert torch.isfinite(out).all()
    r.end(0)
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    r.cache.close()
