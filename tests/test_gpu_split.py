"""Sequence split of a decode step over KV entries (needs a GPU).

hw_concurrent_attention_range attends over a range of every problem's entries (segment order:
common segments in commit order, then the workers' blocks by id) and returns normalised
partials with their log-sum-exp; hw_merge_attention merges such parts.  Every part is compared
with the oracle's attention over the same entries, and the merged parts with the oracle's
attention over the whole view (1e-2 max-abs, the parity tolerance), through both kernels, with
cuts inside tiles, pages and worker blocks, commits, several problems and cache layouts.
"""
import dataclasses

import numpy as np
import pytest

import workload as wl

pytestmark = pytest.mark.gpu

TOL = 1e-2
# A part can hold only a few keys of a view (a range that cuts a worker block, or one a layout
# mostly hides), and then the bf16 roundings do not average out: the P.V product takes P in bf16
# (relative 2^-9 per weight) while the sum is kept in fp32, and the keys and the rotated query
# are bf16 as well, so a part's output can be off by about 2^-8 * max|v| (|v| < 4.5 for these
# N(0,1) values) = 0.018.  Parts are therefore compared at 2e-2; the merged result and the
# attention over the whole view, where many keys contribute, keep the parity tolerance 1e-2.
PART_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from shared_kv_concurrent_gb300.build import build
    build()


def _parts(totals, cuts_per_problem):
    """Ranges [k][P][2] from interior cut points per problem (clipped to the problem's total)."""
    k = len(cuts_per_problem[0]) + 1
    out = []
    for i in range(k):
        row = []
        for p, n in enumerate(totals):
            edges = [0] + [min(int(x), n) for x in cuts_per_problem[p]] + [n]
            row.append((edges[i], max(edges[i], edges[i + 1])))
        out.append(row)
    return np.asarray(out, dtype=np.int64)


def run_split(w, steps, cuts_fn, bernoulli=None, regular_after=True):
    """Decode steps of ``w``; in each, the attention split into ranges and merged on the device,
    compared with the oracle; then the regular call and the step end."""
    import torch
    import gpu_cases as G
    from oracle import attention as A
    from oracle import run as orun
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    r = WorkloadRunner(w)
    c = orun.prefill(w)
    P, W, Hq, D = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim
    worst = 0.0
    for step in range(steps):
        inputs = r.step_inputs(step)
        r.append(inputs)
        orun.append_step(c, w, step)
        q = inputs[2][0]
        qo = orun.query(w, 0, step)
        totals = r.cache.entry_totals()
        assert totals == [A.entry_spans(c, p)[1] for p in range(P)]
        ranges = _parts(totals, cuts_fn(totals, step))
        k = ranges.shape[0]
        po = torch.full((k, P, W, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        pl = torch.full((k, P, W, Hq), float("nan"), dtype=torch.float32, device="cuda")
        for i in range(k):
            r.cache.concurrent_attention_range(0, q, ranges[i], po[i], pl[i])
        out = torch.full((P, W, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((P, W, Hq), float("nan"), dtype=torch.float32, device="cuda")
        binding.hw_merge_attention(po, pl, out, binding.HW_OUT_F32, lse)
        torch.cuda.synchronize()
        for i in range(k):
            ro, rl = A.method_range(c, 0, qo, ranges[i])
            got_o, got_l = po[i].cpu().numpy(), pl[i].cpu().numpy()
            fin = np.isfinite(rl)
            assert np.array_equal(np.isfinite(got_l), fin), (step, i)
            assert np.abs(got_l[fin] - rl[fin]).max(initial=0.0) <= TOL, (step, i)
            err = float(np.abs(got_o - ro).max())
            worst = max(worst, err)
            assert err <= PART_TOL, (step, i, ranges[i].tolist(), err)
        ref, ref_lse = A.method(c, 0, qo)
        err = float(np.abs(out.cpu().numpy() - ref).max())
        worst = max(worst, err)
        assert err <= TOL, (step, err)
        gl = lse.cpu().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin)
        assert np.abs(gl[fin] - ref_lse[fin]).max(initial=0.0) <= TOL
        if regular_after:
            reg = torch.full((P, W, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
            r.attend(inputs, [reg], None, "f32")
            torch.cuda.synchronize()
            assert np.abs(reg.cpu().numpy() - ref).max() <= TOL
        fin_mask = wl.finished_mask(w, step, bernoulli)
        r.end(step, fin_mask)
        c.step_end(fin_mask)
        G.dev_tables_equal(r, c)
    G.check_pools(r, c, 0, 64)
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    r.cache.close()
    return worst


def test_two_way_split_tensor_cores():
    """8 workers, 64 rows per KV head: the common block cut inside a tile, then inside a page
    boundary's tile, over three steps."""
    w = dataclasses.replace(wl.c4(), common_len=(3001,),
                            worker_len=((0, 1, 127, 128, 129, 255, 257, 600),), steps=4)
    cuts = [lambda t: [[1500]], lambda t: [[256 + 77]], lambda t: [[t[0] // 2]]]
    run_split(w, 3, lambda t, s: cuts[s](t))


def test_three_way_split_inside_worker_blocks_with_commits():
    """Cuts inside the worker blocks (entries past the common block), one part empty in some
    steps, with random commits moving blocks into the common history between steps."""
    w = dataclasses.replace(wl.c4(), num_workers=4, common_len=(900,),
                            worker_len=((130, 0, 257, 40),), steps=6)
    run_split(w, 5, lambda t, s: [[900 + 65, max(900 + 66, t[0] - 3 - s)]], bernoulli=0.4)


def test_split_cuda_core_kernel():
    """2 workers x 4 heads per KV head (8 rows): the CUDA-core kernel, four parts."""
    w = dataclasses.replace(wl.tiny(), steps=4)
    run_split(w, 3, lambda t, s: [[100, 513 + s, 600]], bernoulli=0.5)


def test_split_several_problems_step_wise_layout():
    """Two problems cut at different places, in the step-wise layout (other workers' blocks
    hidden), so a range can hold entries that some workers do not see at all."""
    w = dataclasses.replace(wl.c5(), num_problems=2, common_len=(700, 1300),
                            worker_len=((9, 0, 130, 20), (3, 5, 0, 1)), steps=4,
                            layout="step_wise", commit_steps=(1,))
    run_split(w, 3, lambda t, s: [[650 + 10 * s], [t[1] - 7]])


def test_split_contiguous_cache():
    w = dataclasses.replace(wl.c2(), common_len=(1000,), worker_len=((130, 70),), page_size=1280,
                            steps=3)
    run_split(w, 2, lambda t, s: [[333, 1000 + 129]])


def test_merge_kernel_against_the_oracle_merge():
    """The merge alone: random normalised parts (some rows empty in some parts, one row empty in
    all), bf16 and fp32 output, one part (the identity)."""
    import torch
    from oracle import attention as A
    from shared_kv_concurrent_gb300 import binding
    g = np.random.default_rng(3)
    for n, rows, D in ((3, 37, 128), (1, 8, 64), (5, 200, 128)):
        outs = g.standard_normal((n, rows, D)).astype(np.float32)
        lses = (g.standard_normal((n, rows)) * 4).astype(np.float32)
        lses[g.random((n, rows)) < 0.2] = -np.inf
        lses[:, 0] = -np.inf
        ro, rl = A.merge_parts(outs.astype(np.float64), lses.astype(np.float64))
        po, pl = torch.from_numpy(outs).cuda(), torch.from_numpy(lses).cuda()
        for dt, tol in ((binding.HW_OUT_F32, 1e-5), (binding.HW_OUT_BF16, 1e-2)):
            out = torch.full((rows, D), float("nan"), device="cuda",
                             dtype=torch.float32 if dt == binding.HW_OUT_F32 else torch.bfloat16)
            lse = torch.full((rows,), float("nan"), device="cuda")
            binding.hw_merge_attention(po, pl, out, dt, lse)
            torch.cuda.synchronize()
            assert np.abs(out.float().cpu().numpy() - ro).max() <= tol * max(1.0, np.abs(ro).max())
            gl = lse.cpu().numpy()
            assert np.array_equal(np.isfinite(gl), np.isfinite(rl))
            fin = np.isfinite(rl)
            assert np.abs(gl[fin] - rl[fin]).max() <= 1e-5
            assert np.all(out[0].float().cpu().numpy() == 0)


def test_range_and_merge_refusals():
    import torch
    from shared_kv_concurrent_gb300 import HogwildCache, HogwildError, binding
    c = HogwildCache.from_workload(wl.tiny())
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 2, 8, 64, device="cuda")
    lse = torch.zeros(1, 2, 8, device="cuda")
    for bad in ([[5, 4]], [[-1, 3]]):
        with pytest.raises(HogwildError) as e:
            binding.hw_concurrent_attention_range(c.ctx, 0, q, bad, out, lse)
        assert e.value.status == binding.HW_ERR_INVALID_ARG
    with pytest.raises(HogwildError) as e:
        binding.hw_concurrent_attention_range(c.ctx, 0, q, [[0, 3]], out, None)
    assert e.value.status == binding.HW_ERR_INVALID_ARG
    po = torch.zeros(2, 4, 6, device="cuda")                 # head_dim 6: not a multiple of 4
    with pytest.raises(HogwildError) as e:
        binding.hw_merge_attention(po, torch.zeros(2, 4, device="cuda"), torch.zeros(4, 6, device="cuda"),
                                   binding.HW_OUT_F32)
    assert e.value.status == binding.HW_ERR_INVALID_ARG
    c.close()
