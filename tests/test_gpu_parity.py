"""CUDA path against the fp64 oracle, element by element, through the C ABI (needs a GPU).

Sizes span several tiles and pieces with ragged tails; the full 32K-common, 8-worker workload
runs once in the launch configuration the benchmark times.
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


def case(name):
    import gpu_cases as G
    return G


def test_tiny_paged_with_commits():
    import gpu_cases as G
    G.run_case(wl.tiny(), steps=4, bernoulli=0.5)


def test_tiny_contiguous():
    import gpu_cases as G
    G.run_case(wl.tiny(contiguous=True), steps=3)


def test_tiny_bf16_output():
    import gpu_cases as G
    G.run_case(wl.tiny(), steps=2, out_dtype="bf16", pools=False)


def test_w2_contiguous_scaled():
    import gpu_cases as G
    w = G.small(wl.c2(), common_len=(1000,), worker_len=((130, 70),), page_size=1280, steps=3)
    G.run_case(w, steps=3)


def test_full_size_w2_contiguous_36_units_per_group():
    """The 2-worker workload at full size: 288 one-tile units, 36 per (problem, KV head), more
    than one merge warp keeps in flight (two warps share each query row)."""
    import gpu_cases as G
    w = G.small(wl.c2(), steps=3)
    G.run_case(w, steps=2, bernoulli=0.5)


def test_one_kv_head_many_units_cuda_core_and_tensor_cores():
    """One KV head, so every unit of the step belongs to one group (well over 40: four merge
    warps per query row, each folding two batches): 10 rows (CUDA-core kernel) and 64 rows
    (tensor-core kernel)."""
    import gpu_cases as G
    w = G.small(wl.c4(), num_workers=2, num_q_heads=5, num_kv_heads=1, common_len=(20000,),
                worker_len=((300, 77),), steps=3)
    G.run_case(w, steps=2, bernoulli=0.5)
    w = G.small(wl.c4(), num_q_heads=8, num_kv_heads=1, common_len=(30000,),
                worker_len=((0, 1, 127, 128, 129, 255, 257, 600),), steps=3)
    G.run_case(w, steps=2)


def test_w8_paged_permuted_ragged():
    import gpu_cases as G
    w = G.small(wl.c4(), common_len=(3001,), worker_len=((0, 1, 127, 128, 129, 255, 257, 600),),
                steps=3)
    G.run_case(w, steps=3, bernoulli=0.3)


def test_batch_of_problems_with_commits():
    import gpu_cases as G
    w = G.small(wl.c5(), num_problems=3, common_len=(700, 2500, 1300),
                worker_len=((0, 300, 17, 256), (5, 0, 0, 129), (511, 1, 64, 200)), steps=4,
                commit_steps=(1,))
    G.run_case(w, steps=4)


def test_multi_layer():
    import gpu_cases as G
    w = G.small(wl.c3(), num_layers=3, common_len=(2000,), worker_len=((0, 700, 33, 1024),),
                steps=2)
    G.run_case(w, steps=2)


def test_head_dim_64_no_gqa():
    import gpu_cases as G
    w = G.small(wl.tiny(), num_q_heads=4, num_kv_heads=4, num_workers=3, common_len=(300,),
                worker_len=((10, 0, 140),), steps=2)
    G.run_case(w, steps=2, bernoulli=0.5)


def test_head_dim_64_tensor_cores():
    import gpu_cases as G
    w = G.small(wl.tiny(), num_workers=4, num_q_heads=16, num_kv_heads=2, common_len=(700,),
                worker_len=((0, 129, 64, 300),), steps=3)
    G.run_case(w, steps=3, bernoulli=0.5)


def test_single_worker_is_ordinary_decode_on_both_kernels():
    """W = 1, the degenerate case: the view is the common history then the worker's own block,
    i.e. ordinary RoPE decode attention; the worker commits every other step, so its blocks
    keep moving into the history.  8 rows per KV head (CUDA-core kernel) and 16 (tensor cores)."""
    import gpu_cases as G
    for H_q in (16, 32):
        w = G.small(wl.tiny(), num_workers=1, num_q_heads=H_q, num_kv_heads=2,
                    common_len=(900,), worker_len=((130,),), steps=5, commit_steps=(0, 2))
        G.run_case(w, steps=5)


def test_max_rows_128():
    import gpu_cases as G
    w = G.small(wl.c4(), num_workers=16, common_len=(600,),
                worker_len=(tuple(range(0, 160, 10)),), random_page_order=False, steps=2)
    G.run_case(w, steps=2, pools=False)


def test_full_size_w8_common32768():
    """The benchmark workload itself: 32768 common tokens, 8 worker blocks of 128..2048."""
    import gpu_cases as G
    w = G.small(wl.c4(), steps=1)
    G.run_case(w, steps=1, pool_sample=64)


@pytest.mark.parametrize("layout", ["combined", "step_wise", "contiguous", "no_sync"])
def test_cache_layouts_with_commits(layout):
    """Every cache layout (views differ, kernels do not): 4 workers, random commits, so the
    views mix the prompt, committed paragraphs of several writers and live blocks."""
    import gpu_cases as G
    w = G.small(wl.c4(), num_workers=4, common_len=(900,), worker_len=((130, 0, 257, 40),),
                steps=6, layout=layout)
    G.run_case(w, steps=6, bernoulli=0.4)


def test_multi_query_paragraph_header():
    """After a step, two workers append a multi-token header and the others one token; every
    appended token is a query (tensor-core path, 112 query rows of one KV head)."""
    import gpu_cases as G
    w = G.small(wl.c4(), common_len=(1500,), worker_len=((0, 300, 17, 256, 129, 1, 600, 40),),
                steps=3)
    n_new = [[0, 5, 1, 1, 3, 1, 1, 1, 1]]
    G.run_mq_case(w, n_new, [row[1:] for row in n_new], finished=np.array([[0, 1, 0, 0, 1, 0, 0, 0]], np.uint8))


def test_multi_query_older_tokens_and_layouts():
    """Queries that reach back past this step's tokens, in two layouts and two problems."""
    import gpu_cases as G
    for layout in ("combined", "step_wise"):
        w = G.small(wl.c5(), num_problems=2, common_len=(700, 1300),
                    worker_len=((9, 0, 130, 20), (3, 5, 0, 1)), steps=3, layout=layout)
        G.run_mq_case(w, [[0, 1, 1, 1, 1], [2, 1, 1, 0, 1]], [[4, 0, 2, 1], [1, 6, 0, 2]],
                      seed=1)


def test_multi_query_cuda_core_path():
    """Few rows per KV head (2 workers x 4 heads): the CUDA-core kernel with the causal cut."""
    import gpu_cases as G
    w = G.small(wl.tiny(), common_len=(300,), worker_len=((70, 5),), steps=3)
    G.run_mq_case(w, [[0, 3, 1]], [[3, 2]], seed=2)


def test_commits_compaction_then_header_prefill():
    """Decode steps with random commits, a compaction of the committed paragraphs, then a step
    in which two workers prefill a header and attend causally to it -- the inference flow of
    section 8 end to end, on a paged two-layer cache in the step-wise layout."""
    import gpu_cases as G
    w = G.small(wl.c5(), num_problems=2, num_layers=2, common_len=(600, 900),
                worker_len=((40, 0, 130, 7), (12, 300, 1, 0)), steps=12,
                commit_steps=tuple(range(12)), layout="step_wise")
    G.run_mq_case(w, [[0, 4, 1, 1, 1], [2, 1, 6, 1, 1]], [[4, 1, 1, 1], [1, 6, 1, 1]], seed=3,
                  pre_steps=6, bernoulli=0.5, compact=[(0, 0, 5), (1, 1, 4)], max_segments=48)


def test_multi_query_head_dim_64_tensor_cores():
    """The causal cut and the row map on the D = 64 tensor-core kernel."""
    import gpu_cases as G
    w = G.small(wl.tiny(), num_workers=4, num_q_heads=16, num_kv_heads=2, common_len=(700,),
                worker_len=((0, 129, 64, 300),), steps=3)
    G.run_mq_case(w, [[0, 3, 1, 2, 1]], [[3, 1, 2, 4]], seed=4)


def test_multi_query_count_past_the_block_is_refused():
    import torch
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    import gpu_cases as G
    w = G.small(wl.c4(), common_len=(500,), worker_len=((20,) * 8,), steps=2)
    r = WorkloadRunner(w)
    n_q = np.full((1, 8), 1, np.int32)
    n_q[0, 0] = 21                                  # more than the block holds
    q = torch.zeros(28, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(28, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.HogwildError) as e:
        r.cache.concurrent_attention_mq(0, q, n_q, out)
    assert e.value.status == binding.HW_ERR_INVALID_ARG
    n_q[0, 0] = -1
    with pytest.raises(binding.HogwildError) as e:
        r.cache.concurrent_attention_mq(0, q, n_q, out)
    assert e.value.status == binding.HW_ERR_INVALID_ARG
    r.cache.close()


def test_multi_query_rows_split_over_several_launches():
    """More query rows than one 128-row tile: 8 workers x G 8 with 3 or 4 tokens each (200
    rows in one problem), two problems whose parts differ in number, one worker's 40 tokens
    over three launches (its tokens cut inside the worker: the causal offsets of the later
    ones), and a CUDA-core case; every token's output, at its own row, against the oracle."""
    import gpu_cases as G
    w = G.small(wl.c4(), common_len=(1500,), worker_len=((0, 300, 17, 256, 129, 1, 600, 40),),
                steps=3)
    n_new = [[0, 3, 3, 3, 3, 3, 3, 3, 3]]
    n_q = [[3, 3, 3, 3, 4, 3, 3, 3]]                # 25 tokens x 8 = 200 rows: two launches
    G.run_mq_case(w, n_new, n_q)
    w = G.small(wl.c5(), num_problems=2, num_q_heads=64, common_len=(700, 1300),
                worker_len=((9, 0, 130, 20), (3, 5, 0, 1)), steps=3)
    # G 8: 16 tokens per launch; problem 0: 20 tokens (two parts), problem 1: 9 (one part)
    G.run_mq_case(w, [[0, 5, 5, 5, 5], [0, 3, 3, 0, 3]], [[5, 5, 5, 5], [3, 3, 0, 3]])
    w = G.small(wl.c2(), common_len=(1000,), worker_len=((130, 70),), page_size=1280, steps=3)
    # G 5: 25 tokens per launch; 20 + 15 tokens: two launches, the CUDA-core kernel
    G.run_mq_case(w, [[0, 3, 3]], [[20, 15]])
    # one worker's 40 tokens (320 rows at G 8) and a neighbour's 3: three launches (steps=8
    # leaves room in the position table for the 47 appended tokens)
    w = G.small(wl.c4(), common_len=(900,), worker_len=((0, 300, 17, 256, 129, 1, 600, 40),),
                steps=8)
    G.run_mq_case(w, [[0, 1, 40, 1, 1, 1, 1, 1, 1]], [[1, 40, 3, 0, 0, 1, 0, 2]])
    # the CUDA-core kernel: 60 tokens of one worker at G 5 (three launches of at most 25)
    w = G.small(wl.c2(), common_len=(1000,), worker_len=((130, 70),), page_size=1280, steps=3)
    G.run_mq_case(w, [[0, 3, 3]], [[60, 2]])


def test_compaction_policy_between_steps():
    """The library's compaction policy after every step end (more than two paragraphs: merge
    them), with random commits, in the combined layout (all paragraphs into one segment) and
    the contiguous one (runs of one writer): outputs, tables and re-rotated pools against the
    oracle, which applies the merges the policy states."""
    import gpu_cases as G
    for layout in ("combined", "contiguous"):
        w = G.small(wl.c5(), num_problems=2, common_len=(700, 300),
                    worker_len=((9, 0, 130, 20), (3, 5, 0, 1)), steps=8, layout=layout)
        G.run_case(w, steps=7, bernoulli=0.5, compact_auto=2, max_segments=256)


def test_compaction_between_steps():
    """Commits build up committed segments; compactions merge ranges of them (the prompt with
    the first paragraphs, then later paragraphs) and the following steps attend to the merged
    segments: outputs, tables, free list and re-rotated pools against the oracle."""
    import gpu_cases as G
    w = G.small(wl.c5(), num_problems=2, common_len=(700, 300), worker_len=((130, 0, 257, 40),
                (5, 90, 0, 200)), steps=8, num_layers=2,
                commit_steps=tuple(range(8)))    # (page budget for up to one commit a step)
    G.run_case(w, steps=8, bernoulli=0.4,
               compact_after={2: [(0, 0, 3), (1, 1, 4)], 5: [(0, 1, 6), (1, 0, 9)]})


def test_compaction_contiguous_cache_and_refusals():
    import gpu_cases as G
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    w = G.small(wl.c2(), common_len=(1000,), worker_len=((130, 70),), page_size=2048, steps=4,
                commit_steps=(0, 1, 2, 3))     # (page budget for a commit every step)
    G.run_case(w, steps=4, bernoulli=0.6, compact_after={1: [(0, 0, 4)], 2: [(0, 0, 4)]},
               max_segments=32)         # (each commit and each compaction adds a segment)
    r = WorkloadRunner(w)
    for args in ((0, 0, 1), (0, 1, 2), (1, 0, 2)):   # too few, past the list, no such problem
        with pytest.raises(binding.HogwildError) as e:
            r.cache.compact_segments(*args)
        assert e.value.status == binding.HW_ERR_INVALID_ARG
    r.cache.close()


def test_full_size_w4_common16384_64_layers():
    """All 64 layers run on the device; the oracle computes the first two and the last layer
    (the tables are shared by every layer, the pools are not)."""
    import gpu_cases as G
    G.run_case(wl.c3(), steps=2, layer_ids=(0, 1, 63), pool_sample=64)


def test_full_size_16_problems_200_steps_with_commits():
    """Every step and every commit (after steps 63, 127, 191) runs on the device, the tables are
    compared after each step end, the outputs on both sides of each commit and at the ends."""
    import gpu_cases as G
    w = wl.c5()
    G.run_case(w, steps=w.steps, check_steps={0, 63, 64, 127, 128, 191, 192, 199},
               pool_sample=64)


def test_empty_view_gives_zero_and_minus_inf():
    import torch
    from shared_kv_concurrent_gb300 import HogwildCache
    w = G_small_empty()
    c = HogwildCache.from_workload(w)
    q = torch.randn(1, 2, 8, 64, device="cuda").to(torch.bfloat16)
    lse = torch.zeros(1, 2, 8, device="cuda")
    out = c.concurrent_attention(0, q, out_dtype="f32", lse=lse)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)
    c.close()


def G_small_empty():
    import dataclasses
    return dataclasses.replace(wl.tiny(), common_len=(0,), worker_len=((0, 0),))


@pytest.mark.parametrize("H_q,kid", [(16, 4), (4, 2)])      # tensor-core, CUDA-core kernel
def test_plan_wait_times_out_and_the_context_recovers(H_q, kid):
    """A plan announced with a sequence number that never arrives (host-side injection): the
    attention kernel gives up after its bounded wait, outputs zero and reports a timeout; the
    next calls, outside and inside a step, are correct again."""
    import torch
    import gpu_cases as G
    from oracle import attention as A
    from oracle import run as orun
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner, to_device_bf16
    w = G.small(wl.tiny(), num_workers=4, num_q_heads=H_q, num_kv_heads=2, common_len=(300,),
                worker_len=((5, 0, 130, 64),), steps=2)
    r = WorkloadRunner(w)
    c = orun.prefill(w)
    P, W, D = w.num_problems, w.num_workers, w.head_dim
    zeros = np.zeros((P, W), np.uint8)
    inp = r.step_inputs(0)
    r.append(inp)
    orun.append_step(c, w, 0)
    out = torch.empty(P, W, H_q, D, device="cuda")
    r.attend(inp, [out], None, "f32")
    r.end(0, zeros)
    c.step_end(zeros)
    assert r.cache.check_device_errors()[0] == binding.HW_OK
    # outside a step: the call uploads its own plan, which is the one that expires
    q = to_device_bf16(wl.step_q(w, 0, 1))
    lse = torch.empty(P, W, H_q, device="cuda")
    binding.hw_debug_expire_plans(r.cache.ctx, 1)
    out.fill_(float("nan"))
    r.cache.concurrent_attention(0, q, out, "f32", lse)
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_ERR_DEVICE_TIMEOUT and info[1] == kid, (st, info)
    assert torch.all(out == 0) and torch.all(torch.isinf(lse) & (lse < 0))
    ref, ref_lse = A.method(c, 0, orun.query(w, 0, 1))
    r.cache.concurrent_attention(0, q, out, "f32", lse)
    assert r.cache.check_device_errors()[0] == binding.HW_OK
    assert np.abs(out.cpu().numpy() - ref).max() <= G.TOL
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= G.TOL
    # and a whole decode step after it
    inp = r.step_inputs(1)
    r.append(inp)
    orun.append_step(c, w, 1)
    r.attend(inp, [out], [lse], "f32")
    ref, ref_lse = A.method(c, 0, orun.query(w, 0, 1))
    assert r.cache.check_device_errors()[0] == binding.HW_OK
    assert np.abs(out.cpu().numpy() - ref).max() <= G.TOL
    r.end(1, zeros)
    c.step_end(zeros)
    G.dev_tables_equal(r, c)
    r.cache.close()


def test_last_rope_position_then_the_position_limit():
    """Views that reach the RoPE table's last row are exact; the append that would pass it is
    refused with nothing changed, and attention afterwards still matches."""
    import dataclasses
    import torch
    import gpu_cases as G
    from oracle import attention as A
    from oracle import run as orun
    from shared_kv_concurrent_gb300 import HogwildError, binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner, to_device_bf16
    w = G.small(wl.tiny(), steps=3)
    limit = w.view_tokens(1)                     # view length after step 1's append

    @dataclasses.dataclass(frozen=True)
    class Limited(type(w)):
        def max_position(self) -> int:
            return limit

    r = WorkloadRunner(Limited(**{f.name: getattr(w, f.name) for f in dataclasses.fields(w)}))
    c = orun.prefill(w)
    P, W, Hq, D = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim
    zeros = np.zeros((P, W), np.uint8)
    out = torch.empty(P, W, Hq, D, device="cuda")
    for step in range(2):
        inp = r.step_inputs(step)
        r.append(inp)
        orun.append_step(c, w, step)
        r.attend(inp, [out], None, "f32")
        ref, _ = A.method(c, 0, orun.query(w, 0, step))
        assert np.abs(out.cpu().numpy() - ref).max() <= G.TOL, step
        r.end(step, zeros)
        c.step_end(zeros)
    assert max(c.view(p, wk)[-1] for p in range(P) for wk in range(W)) == limit - 1
    with pytest.raises(HogwildError) as e:
        r.append(r.step_inputs(2))
    assert e.value.status == binding.HW_ERR_CAPACITY
    G.dev_tables_equal(r, c)
    q = to_device_bf16(wl.step_q(w, 0, 1))
    r.cache.concurrent_attention(0, q, out, "f32")
    ref, _ = A.method(c, 0, orun.query(w, 0, 1))
    assert np.abs(out.cpu().numpy() - ref).max() <= G.TOL
    assert r.cache.check_device_errors()[0] == binding.HW_OK
    r.cache.close()


def test_many_multi_query_calls_inside_one_step():
    """More several-query calls inside one step than the context has plan slots: the step's own
    plan (its append runs and decode attention plan) must survive them."""
    import torch
    import gpu_cases as G
    from oracle import attention as A
    from oracle import run as orun
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner, to_device_bf16
    w = G.small(wl.tiny(), steps=2)
    r = WorkloadRunner(w)
    c = orun.prefill(w)
    P, W, Hq, D = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim
    inputs = r.step_inputs(0)
    r.append(inputs)
    orun.append_step(c, w, 0)
    q = orun.query(w, 0, 0)
    ref, _ = A.method(c, 0, q)
    n_q = np.ones((P, W), np.int32)                 # each worker's newest token: the decode query
    qd = to_device_bf16(wl.step_q(w, 0, 0).reshape(P * W, Hq, D))
    out = torch.empty(P * W, Hq, D, device="cuda")
    for _ in range(70):                              # more than the at most 32 plan slots
        r.cache.concurrent_attention_mq(0, qd, n_q, out, "f32")
    torch.cuda.synchronize()
    assert np.abs(out.cpu().numpy().reshape(P, W, Hq, D) - ref).max() <= G.TOL
    outs = [torch.empty(P, W, Hq, D, device="cuda")]
    r.attend(inputs, outs, None, "f32")             # the step's own plan
    torch.cuda.synchronize()
    assert np.abs(outs[0].cpu().numpy() - ref).max() <= G.TOL
    zeros = np.zeros((P, W), np.uint8)
    r.end(0, zeros)
    c.step_end(zeros)
    G.dev_tables_equal(r, c)
    G.check_pools(r, c, 0)
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    r.cache.close()


def test_protocol_errors_leave_state_unchanged():
    import torch
    from shared_kv_concurrent_gb300 import HogwildCache, HogwildError, binding
    w = wl.tiny()
    c = HogwildCache.from_workload(w)
    k = torch.zeros(2, 2, 64, dtype=torch.bfloat16, device="cuda")
    n = np.array([[0, 1, 1]], np.int32)
    c.append_kv(0, n, k, k)
    with pytest.raises(HogwildError) as e:
        c.append_kv(0, n, k, k)                      # same layer twice in one step
    assert e.value.status == binding.HW_ERR_INVALID_ARG
    c.step_end(None)
    before = c.tables()
    big = np.array([[10 ** 6, 0, 0]], np.int32)
    kb = torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(HogwildError) as e:
        c.append_kv(0, big, kb, kb)
    assert e.value.status in (binding.HW_ERR_OUT_OF_PAGES, binding.HW_ERR_CAPACITY)
    assert c.tables() == before
    st, info = c.check_device_errors()
    assert st == binding.HW_OK, info
    c.close()


def test_out_of_pages_reported():
    import dataclasses
    import torch
    from shared_kv_concurrent_gb300 import HogwildCache, HogwildError, binding, config_for
    cfg = config_for(num_problems=1, num_workers=2, num_layers=1, num_q_heads=8, num_kv_heads=2,
                     head_dim=64, page_size=128, num_pages=3, max_position=4096, rope_theta=1e4)
    c = HogwildCache(cfg)
    k = torch.zeros(300, 2, 64, dtype=torch.bfloat16, device="cuda")
    c.append_kv(0, np.array([[300, 0, 0]], np.int32), k, k)       # 3 pages
    c.step_end(None)
    before = c.tables()
    with pytest.raises(HogwildError) as e:
        c.append_kv(0, np.array([[0, 1, 0]], np.int32), k[:1], k[:1])
    assert e.value.status == binding.HW_ERR_OUT_OF_PAGES
    assert c.tables() == before
    c.close()
    del dataclasses


def test_deterministic_bitwise():
    import torch
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    import gpu_cases as G
    w = G.small(wl.c4(), common_len=(2000,), worker_len=((5, 300, 0, 77, 128, 256, 1, 999),),
                steps=1)
    r = WorkloadRunner(w)
    inp = r.step_inputs(0)
    r.append(inp)
    o1 = [torch.empty(1, 8, 64, 128, dtype=torch.float32, device="cuda")]
    o2 = [torch.empty_like(o1[0])]
    r.attend(inp, o1, None, "f32")
    r.attend(inp, o2, None, "f32")
    torch.cuda.synchronize()
    assert torch.equal(o1[0].view(torch.int32), o2[0].view(torch.int32))
    r.cache.close()


def test_multi_token_appends_fused_and_deferred():
    """Tensor-core context (64 query rows): a step appending 17 tokens per worker (append
    kernel), one appending 16 (written inside the attention kernel), one whose appends no
    attention call writes (the step end writes them), then a decode step -- each attended step
    against the oracle, with pools and tables."""
    import torch
    import gpu_cases as G
    from oracle import attention as A
    from oracle import run as orun
    from shared_kv_concurrent_gb300.runner import WorkloadRunner, to_device_bf16
    w = G.small(wl.c4(), common_len=(700,), worker_len=((0, 5, 127, 128, 129, 40, 300, 1),),
                random_page_order=True, steps=40)     # page budget for the 36 extra tokens
    r = WorkloadRunner(w)
    c = orun.prefill(w)
    P, W, Hq, Hkv, D = w.num_problems, w.num_workers, w.num_q_heads, w.num_kv_heads, w.head_dim
    rng = np.random.default_rng(7)

    def bits(*shape):
        return wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))

    for per_worker, common, attend in ((17, 3, True), (16, 0, True), (2, 1, False), (1, 0, True)):
        n = np.zeros((P, W + 1), np.int32)
        n[:, 0] = common
        n[:, 1:] = per_worker
        tot = int(n.sum())
        kb, vb, qb = bits(tot, Hkv, D), bits(tot, Hkv, D), bits(P, W, Hq, D)
        kd, vd, qd = to_device_bf16(kb), to_device_bf16(vb), to_device_bf16(qb)
        r.cache.append_kv(0, n, kd, vd)
        c.append(0, n, orun.bf16(kb), orun.bf16(vb))
        if attend:
            out = torch.full((P, W, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
            r.cache.concurrent_attention(0, qd, out, "f32")
            torch.cuda.synchronize()
            ref, _ = A.method(c, 0, orun.bf16(qb).astype(np.float64))
            err = float(np.abs(out.cpu().numpy() - ref).max())
            assert err <= G.TOL, (per_worker, err)
        fin = np.zeros((P, W), np.uint8)
        r.cache.step_end(fin)
        c.step_end(fin)
        torch.cuda.synchronize()
        G.check_pools(r, c, 0)
        G.dev_tables_equal(r, c)
    from shared_kv_concurrent_gb300 import binding
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    r.cache.close()


def test_readme_example():
    """The usage example of the README runs as written (and matches the oracle)."""
    import torch
    from oracle import attention as A
    from oracle.cache import HogwildCache as OracleCache
    from shared_kv_concurrent_gb300 import HogwildCache, config_for
    g = torch.Generator().manual_seed(7)
    k_new = torch.randn(8, 8, 128, generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn(8, 8, 128, generator=g).to(torch.bfloat16).cuda()
    q = torch.randn(1, 8, 64, 128, generator=g).to(torch.bfloat16).cuda()
    cfg = config_for(num_problems=1, num_workers=8, num_layers=1, num_q_heads=64, num_kv_heads=8,
                     head_dim=128, page_size=256, num_pages=4096, max_position=1 << 17,
                     rope_theta=1e6)
    cache = HogwildCache(cfg)
    n_new = np.ones((1, 9), np.int32)
    n_new[0, 0] = 0
    cache.append_kv(0, n_new, k_new, v_new)
    out = cache.concurrent_attention(0, q)
    cache.step_end(np.zeros((1, 8), np.uint8))
    torch.cuda.synchronize()
    oc = OracleCache(1, 8, 1, 8, 128, 1e6, 256, 4096)
    oc.append(0, n_new, k_new.float().cpu().numpy(), v_new.float().cpu().numpy())
    ref, _ = A.method(oc, 0, q.float().cpu().numpy())
    assert np.abs(out.float().cpu().numpy() - ref).max() <= 1e-2
    cache.close()


@pytest.mark.parametrize("seed,layout,D,H_q,H_kv,S", [
    (11, "combined", 64, 8, 2, 128), (12, "step_wise", 64, 8, 2, 128),
    (13, "contiguous", 128, 16, 2, 128), (14, "no_sync", 128, 16, 2, 128),
    (15, "combined", 128, 32, 4, 256), (16, "step_wise", 128, 64, 8, 256),
    (17, "contiguous", 64, 16, 4, 256), (18, "combined", 128, 16, 1, 128)])
def test_random_sessions(seed, layout, D, H_q, H_kv, S):
    """Every entry point in seeded random order against the oracle (see run_random_session)."""
    import gpu_cases as G
    _, stats = G.run_random_session(seed, layout=layout, D=D, H_q=H_q, H_kv=H_kv, S=S, steps=14)
    assert stats["decode"] and stats["mq"] and stats["commits"], stats
    assert stats["compacted"] + stats["refused"] > 0, stats
    print(seed, layout, stats)
