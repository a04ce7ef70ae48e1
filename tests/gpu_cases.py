"""Shared driver of the GPU parity tests: run a workload through the library and the oracle
side by side and compare every output, table and stored slot."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import workload as wl
from oracle import attention as A
from oracle import run as orun

# Output tolerance: max-abs 1e-2 on bf16 inputs with fp32 accumulation.  The budget: keys are
# stored as bf16 (relative error 2^-9) which perturbs a logit q.k/sqrt(D) of N(0,1) data by
# about 0.004; the bf16 output adds < 0.004 for |o| < 2.
TOL = 1e-2


def dev_tables_equal(runner, cache):
    got = runner.cache.tables()
    exp = cache.tables()
    assert got["common"] == exp["common"], (got["common"], exp["common"])
    assert got["live"] == exp["live"]
    assert got["free_count"] == exp["free_count"]
    assert [tuple(s[:4]) for s in got["segments"]] == [tuple(s[:4]) for s in exp["segments"]]
    assert [list(s[4]) for s in got["segments"]] == [list(s[4]) for s in exp["segments"]]
    for p in range(cache.P):
        for w in range(cache.W):
            e, iq = cache.view(p, w)
            ge, giq = runner.cache.view(p, w)
            assert giq == iq and [tuple(x) for x in ge] == [tuple(x) for x in e]


def check_pools(runner, cache, layer, max_tokens_per_seg=None, dev_layer=None, rerotated=None):
    """Stored keys within 1 bf16 ulp of the fp64 rotation; values bit-exact; at the oracle's
    (page, slot) of every token -- so page addressing is checked bit-exactly too.

    ``layer`` indexes the oracle cache, ``dev_layer`` (default: the same) the library's."""
    import torch
    kp, vp = runner.cache.pools(layer if dev_layer is None else dev_layer)
    kb = kp.view(torch.int16).cpu().numpy().view(np.uint16)
    vb = vp.view(torch.int16).cpu().numpy().view(np.uint16)
    for sid, seg in enumerate(cache.segments):
        n = seg.visible
        if n == 0:
            continue
        js = np.arange(n)
        if max_tokens_per_seg and n > max_tokens_per_seg:
            js = np.unique(np.concatenate([js[:8], js[-8:], np.random.default_rng(sid).choice(
                n, max_tokens_per_seg, replace=False)]))
        sk = seg.stored_k(layer)[js]
        rv = seg.raw_v(layer)[js]
        slots = [cache.slot_of(sid, int(j)) for j in js]
        pg = np.array([s[0] for s in slots])
        sl = np.array([s[1] for s in slots])
        gk = wl.bf16_bits_to_f32(kb[pg, :, sl, :]).astype(np.float64)   # [n][H_kv][D]
        gv = vb[pg, :, sl, :]
        ev = wl.f32_to_bf16_bits(rv.astype(np.float32))
        # Stored key = bf16(x1 c - x2 s) computed in fp32: rounding to bf16 costs at most half
        # an ulp (unit roundoff 2^-8 relative) and the fp32 products, the fp32 cos/sin table and
        # the cancellation at most a few 2^-24 of the pair's magnitude, which dominates when the
        # rotated value nearly cancels.
        rk = seg.raw_k(layer)[js]
        half = rk.shape[-1] // 2
        pair = np.abs(rk[..., :half]) + np.abs(rk[..., half:])
        pair = np.concatenate([pair, pair], axis=-1)
        bound = 2.0 ** -8 * np.abs(sk) + 2.0 ** -21 * pair
        if rerotated and sid in rerotated:
            # A compacted key was rounded to bf16 at its block-local position, then turned by
            # its offset in fp32 and rounded again, once per compaction it went through: each
            # earlier rounding error (half an ulp of each element) is mixed across the pair by
            # the rotations after it.
            bound = 2.0 ** -8 * np.abs(sk) + rerotated[sid] * 2.0 ** -8 * pair
        excess = np.abs(gk - sk) - bound
        assert excess.max() <= 0, (sid, float(np.abs(gk - sk).max()), float(excess.max()))
        assert np.array_equal(gv, ev), sid


def run_case(w: wl.Workload, steps: int, out_dtype="f32", bernoulli=None, pools=True,
             pool_sample=None, tol=TOL, layer_ids=None, check_steps=None, compact_after=None,
             max_segments=0, compact_auto=None):
    """Run ``steps`` decode steps on both sides; compare tables after every step end.

    ``layer_ids``: the workload layers the oracle computes (default all); the library always
    runs every layer.  ``compact_after``: {step: [(problem, first, count), ...]} compactions
    done on both sides after that step's end (a range that reaches past the common list is
    cut to it).  ``compact_auto``: after every step end the library's compaction policy
    (hw_compact_auto with that max_paragraphs) on the device, and the same merges, as the policy
    states them, on the oracle (at least one merge must happen in the run).  ``check_steps``: the steps whose outputs (and pools) are compared
    (default all) -- the oracle still appends every step, so later steps see the same cache.
    """
    import torch
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner
    r = WorkloadRunner(w, max_segments=max_segments)
    ids = list(range(w.num_layers)) if layer_ids is None else list(layer_ids)
    c = orun.prefill(w, layer_ids=ids)
    dev_tables_equal(r, c)
    worst = 0.0
    P, W, Hq, D = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    rerotated = {}                        # compacted segment -> compactions its keys went through
    auto_merges = 0
    for step in range(steps):
        inputs = r.step_inputs(step)
        r.append(inputs)
        orun.append_step(c, w, step, layer_ids=ids)
        outs = [torch.full((P, W, Hq, D), float("nan"), dtype=dt, device="cuda")
                for _ in range(w.num_layers)]
        lses = [torch.full((P, W, Hq), float("nan"), dtype=torch.float32, device="cuda")
                for _ in range(w.num_layers)]
        r.attend(inputs, outs, lses, out_dtype)
        torch.cuda.synchronize()
        if check_steps is None or step in check_steps:
            for i, layer in enumerate(ids):
                ref, ref_lse = A.method(c, i, orun.query(w, layer, step))
                got = outs[layer].float().cpu().numpy()
                err = np.abs(got - ref).max()
                worst = max(worst, float(err))
                assert err <= tol, (step, layer, err)
                gl = lses[layer].cpu().numpy()
                fin = np.isfinite(ref_lse)
                assert np.array_equal(np.isfinite(gl), fin)
                assert np.abs(gl[fin] - ref_lse[fin]).max() <= tol
                if pools:
                    check_pools(r, c, i, pool_sample, dev_layer=layer, rerotated=rerotated)
        fin = wl.finished_mask(w, step, bernoulli)
        r.end(step, fin)
        c.step_end(fin)
        dev_tables_equal(r, c)
        for p, first, count in (compact_after or {}).get(step, []):
            count = min(count, len(c.common[p]) - first)
            if count < 2:
                continue
            depth = 1 + max(rerotated.get(sid, 0) for sid in c.common[p][first:first + count])
            r.cache.compact_segments(p, first, count)
            rerotated[c.compact(p, first, count)] = depth
            dev_tables_equal(r, c)
        if compact_auto is not None:
            ranges = []
            for p in range(w.num_problems):
                com = c.common[p]
                if len(com) - 1 <= compact_auto:
                    continue
                if w.layout in ("contiguous", "no_sync"):
                    # runs of consecutive paragraphs of one writer
                    i = 1
                    while i < len(com):
                        j = i + 1
                        while j < len(com) and c.segments[com[j]].origin == c.segments[com[i]].origin:
                            j += 1
                        if j - i >= 2:
                            ranges.append((p, i, j - i))
                        i = j
                else:
                    ranges.append((p, 1, len(com) - 1))
            merges = r.cache.compact_auto(compact_auto)
            assert merges == len(ranges), (step, merges, ranges)
            auto_merges += merges
            # the oracle applies them left to right; a merged run leaves one entry behind
            shift = {}
            for p, first, count in ranges:
                first -= shift.get(p, 0)
                depth = 1 + max(rerotated.get(sid, 0) for sid in c.common[p][first:first + count])
                rerotated[c.compact(p, first, count)] = depth
                shift[p] = shift.get(p, 0) + count - 1
            dev_tables_equal(r, c)
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    assert compact_auto is None or auto_merges > 0
    r.cache.close()
    return worst


def small(base: wl.Workload, **kw) -> wl.Workload:
    return dataclasses.replace(base, **kw)


def run_mq_case(w: wl.Workload, n_new, n_q, seed=0, tol=TOL, finished=None, pre_steps=0,
                bernoulli=0.5, compact=(), max_segments=0):
    """One step with a custom append (n_new [P][W+1]) and several causal query tokens per worker
    (n_q [P][W]) through hw_concurrent_attention_mq, against the oracle's method_mq; then the
    step end and one ordinary decode step.  Before it: ``pre_steps`` ordinary decode steps with
    random commits, then the compactions ``compact`` [(problem, first, count)] on both sides."""
    import torch
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner, to_device_bf16
    r = WorkloadRunner(w, max_segments=max_segments)
    c = orun.prefill(w)
    for step in range(pre_steps):
        inputs = r.step_inputs(step)
        r.append(inputs)
        orun.append_step(c, w, step)
        r.attend(inputs, [torch.empty(w.num_problems, w.num_workers, w.num_q_heads, w.head_dim,
                                      dtype=torch.bfloat16, device="cuda")
                          for _ in range(w.num_layers)])
        fin = wl.finished_mask(w, step, bernoulli)
        r.end(step, fin)
        c.step_end(fin)
    rerotated = {}                        # compacted segment -> compactions its keys went through
    for p, first, count in compact:
        count = min(count, len(c.common[p]) - first)
        if count >= 2:
            depth = 1 + max(rerotated.get(sid, 0) for sid in c.common[p][first:first + count])
            r.cache.compact_segments(p, first, count)
            rerotated[c.compact(p, first, count)] = depth
    dev_tables_equal(r, c)
    g = np.random.default_rng(seed)
    n_new = np.asarray(n_new, dtype=np.int32).reshape(w.num_problems, w.num_workers + 1)
    n_q = np.asarray(n_q, dtype=np.int32).reshape(w.num_problems, w.num_workers)
    tot = int(n_new.sum())
    kb = wl.f32_to_bf16_bits(g.standard_normal((tot, w.num_kv_heads, w.head_dim)).astype(np.float32))
    vb = wl.f32_to_bf16_bits(g.standard_normal((tot, w.num_kv_heads, w.head_dim)).astype(np.float32))
    N = int(n_q.sum())
    qb = wl.f32_to_bf16_bits(g.standard_normal((N, w.num_q_heads, w.head_dim)).astype(np.float32))
    worst = 0.0
    kd, vd = to_device_bf16(kb), to_device_bf16(vb)   # read until the step's attention
    for layer in range(w.num_layers):
        r.cache.append_kv(layer, n_new, kd, vd)
        c.append(layer, n_new, orun.bf16(kb), orun.bf16(vb))
    for layer in range(w.num_layers):
        out = torch.full((N, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.float32,
                         device="cuda")
        lse = torch.full((N, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
        r.cache.concurrent_attention_mq(layer, to_device_bf16(qb), n_q, out, "f32", lse)
        torch.cuda.synchronize()
        ref, ref_lse = A.method_mq(c, layer, orun.bf16(qb).astype(np.float64), n_q)
        got = out.cpu().numpy()
        err = float(np.abs(got - ref).max()) if N else 0.0
        worst = max(worst, err)
        assert err <= tol, (layer, err)
        if N:
            assert np.abs(lse.cpu().numpy() - ref_lse).max() <= tol
        check_pools(r, c, layer, 64, rerotated=rerotated)
    fin = np.zeros((w.num_problems, w.num_workers), np.uint8) if finished is None else finished
    r.end(pre_steps, fin)
    torch.cuda.synchronize()
    del kd, vd
    c.step_end(fin)
    dev_tables_equal(r, c)
    # an ordinary decode step afterwards
    nxt = pre_steps + 1
    inputs = r.step_inputs(nxt)
    r.append(inputs)
    orun.append_step(c, w, nxt)
    P, W, Hq, D = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim
    outs = [torch.full((P, W, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
            for _ in range(w.num_layers)]
    r.attend(inputs, outs, None, "f32")
    torch.cuda.synchronize()
    for layer in range(w.num_layers):
        ref, _ = A.method(c, layer, orun.query(w, layer, nxt))
        assert np.abs(outs[layer].cpu().numpy() - ref).max() <= tol
    st, info = r.cache.check_device_errors()
    assert st == binding.HW_OK, info
    r.cache.close()
    return worst


def run_random_session(seed: int, layout="combined", P=2, W=3, H_q=8, H_kv=2, D=64, L=2,
                       S=128, steps=10, tol=TOL):
    """Seeded random use of every entry point against the oracle: appends of 0..3 tokens per
    block (sometimes a long one, which takes the append kernel), decode or multi-query attention
    of every layer, random commits, and compactions of random common ranges (a refusal must
    match on both sides).  Tables after every step end; pools at the end."""
    import torch
    from shared_kv_concurrent_gb300 import HogwildCache, binding, config_for
    from shared_kv_concurrent_gb300.runner import to_device_bf16
    from oracle import cache as OC
    g = np.random.default_rng(seed)
    pages = 2048
    order = g.permutation(pages).astype(np.int32)
    cfg = config_for(num_problems=P, num_workers=W, num_layers=L, num_q_heads=H_q,
                     num_kv_heads=H_kv, head_dim=D, page_size=S, num_pages=pages,
                     max_position=1 << 14, rope_theta=1e4, max_segments=256, layout=layout)
    dev = HogwildCache(cfg, page_order=order)
    c = OC.HogwildCache(P, W, L, H_kv, D, 1e4, S, pages, page_order=order, layout=layout)

    class _R:                               # what dev_tables_equal / check_pools expect
        cache = dev
    r = _R()
    bf = lambda shape: wl.f32_to_bf16_bits(g.standard_normal(shape).astype(np.float32))
    rerotated = {}
    worst = 0.0
    stats = {"decode": 0, "mq": 0, "compacted": 0, "refused": 0, "commits": 0}
    for step in range(steps):
        n_new = g.integers(0, 4, size=(P, W + 1)).astype(np.int32)
        if step == 0 or g.random() < 0.2:
            n_new[g.integers(P), g.integers(W + 1)] += int(g.integers(17, 60))
        tot = int(n_new.sum())
        keep = []
        for layer in range(L):
            kb, vb = bf((tot, H_kv, D)), bf((tot, H_kv, D))
            kd, vd = to_device_bf16(kb), to_device_bf16(vb)
            keep.append((kd, vd))
            dev.append_kv(layer, n_new, kd, vd)
            c.append(layer, n_new, orun.bf16(kb), orun.bf16(vb))
        own = np.array([[c.segments[c.live[p][w]].visible for w in range(W)] for p in range(P)])
        use_mq = g.random() < 0.5
        stats["mq" if use_mq else "decode"] += 1
        if use_mq:
            n_q = np.minimum(own, g.integers(0, 4, size=(P, W))).astype(np.int32)
            while (n_q.sum(axis=1) * (H_q // H_kv)).max() > 128:
                n_q = n_q // 2
        for layer in range(L):
            if use_mq:
                N = int(n_q.sum())
                if N == 0:
                    continue
                qb = bf((N, H_q, D))
                out = torch.full((N, H_q, D), float("nan"), device="cuda")
                lse = torch.full((N, H_q), float("nan"), device="cuda")
                dev.concurrent_attention_mq(layer, to_device_bf16(qb), n_q, out, "f32", lse)
                ref, ref_lse = A.method_mq(c, layer, orun.bf16(qb).astype(np.float64), n_q)
            else:
                qb = bf((P, W, H_q, D))
                out = torch.full((P, W, H_q, D), float("nan"), device="cuda")
                lse = torch.full((P, W, H_q), float("nan"), device="cuda")
                dev.concurrent_attention(layer, to_device_bf16(qb), out, "f32", lse)
                ref, ref_lse = A.method(c, layer, orun.bf16(qb).astype(np.float64))
            torch.cuda.synchronize()
            got, gl = out.cpu().numpy(), lse.cpu().numpy()
            err = float(np.abs(got - ref).max())
            worst = max(worst, err)
            assert err <= tol, (seed, layout, step, layer, use_mq, err)
            fin_ = np.isfinite(ref_lse)
            assert np.array_equal(np.isfinite(gl), fin_)
            assert np.abs(gl[fin_] - ref_lse[fin_]).max(initial=0.0) <= tol
        fin = (g.random((P, W)) < 0.3).astype(np.uint8)
        stats["commits"] += int(fin.sum())
        dev.step_end(fin)
        c.step_end(fin)
        torch.cuda.synchronize()
        del keep
        dev_tables_equal(r, c)
        if g.random() < 0.4:
            p = int(g.integers(P))
            n_common = len(c.common[p])
            if n_common >= 2:
                first = int(g.integers(0, n_common - 1))
                count = int(g.integers(2, n_common - first + 1))
                olds = c.common[p][first:first + count]
                try:
                    sid = c.compact(p, first, count)
                except OC.InvalidArg:
                    with pytest.raises(binding.HogwildError) as e:
                        dev.compact_segments(p, first, count)
                    assert e.value.status == binding.HW_ERR_INVALID_ARG
                    stats["refused"] += 1
                else:
                    dev.compact_segments(p, first, count)
                    stats["compacted"] += 1
                    rerotated[sid] = 1 + max(rerotated.get(s_, 0) for s_ in olds)
                dev_tables_equal(r, c)
    for layer in range(L):
        check_pools(r, c, layer, None, rerotated=rerotated)
    st, info = dev.check_device_errors()
    assert st == binding.HW_OK, info
    dev.close()
    return worst, stats
