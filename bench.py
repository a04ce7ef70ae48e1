"""Benchmark of the Hogwild! concurrent-attention decode step on GB300.

A step is one pass of the whole hot path over one batch of synthetic input: append one new
token per worker (K rotated to its block-local position, bf16 into its page), the concurrent
attention of every worker over its own view (per-block query rotation, split over KV entries,
log-sum-exp merge), and the step end.  Default workload: 1 problem, 8 workers, H_q 64, H_kv 8,
D 128, a 32768-token common block plus 8 worker blocks of 128..2048 tokens in a paged cache
(page 256, seeded random physical page order).

Reported (one JSON line, rank 0):
  value  effective HBM GB/s = algorithmic bytes / device time of K consecutive steps (one
         CUDA event pair), inputs resident in HBM; the steps go in turn to several
         independent caches of the workload, so each step's K/V come from HBM, not L2.  The
         algorithmic bytes count every K/V element once (not once per worker), plus q, out
         and the appended K/V.
  e2e    the same metric through the public API with pinned host buffers
         (hw_decode_step_host): one H2D copy of the step's new K/V and queries, the step, one
         D2H copy of the outputs and a stream synchronize, all inside the timer.
  roofline  the attention kernel's algorithmic bytes / its duration in the timed chain (the
         chained step time x the kernel's share of the step's kernel time, from CUDA events
         around every kernel in a second pass) vs measured HBM; the unchained per-launch figure
         of that pass is reported beside it.
  cpu_baseline  the fp64 oracle on the host cores on a bounded sample of the same workload.
``--impl reference`` times that oracle alone on the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "concurrent-attn effective HBM GB/s (% of peak) and worker-tokens/s per step"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def captured_traffic():
    """DRAM bytes per attention launch from the committed ncu summary, or None if the kernel's
    sources changed since that capture (the summary records their hash)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "attn_tc_kernel_w8_common32768.md")) as f:
            text = f.read()
        rec = text.split("kernel-source-sha256:")[1].split()[0]
        traffic = int(text.split("traffic-bytes-per-launch:")[1].split()[0])
        h = hashlib.sha256()
        for name in ("attn_tc.cu", "tc_ptx.cuh", "hw_internal.h", "hw_device.cuh"):
            with open(os.path.join(ROOT, "shared_kv_concurrent_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        return traffic if h.hexdigest() == rec else None
    except Exception:
        return None


def captured_share():
    """The attention kernel's share of the decode step's kernel time from the committed ncu
    launch list (cold and serialised: a share, not an absolute), or None if the kernel sources
    changed since that list was taken (the summary records their hash)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "launches_w8_common32768_step.md")) as f:
            text = f.read()
        rec = text.split("kernel-source-sha256:")[1].split()[0]
        share = float(text.split("attention-share-of-step:")[1].split()[0])
        h = hashlib.sha256()
        for name in ("attn_tc.cu", "merge.cu", "hw_merge.cuh", "tc_ptx.cuh", "hw_internal.h",
                     "hw_device.cuh"):
            with open(os.path.join(ROOT, "shared_kv_concurrent_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        return share if h.hexdigest() == rec else None
    except Exception:
        return None


def workload_for(name, layout="combined", seed=None):
    """The named workload; another cache layout changes only the views (and the name); another
    master seed redraws the block lengths, the page order and every tensor (and the name)."""
    import dataclasses

    import workload as wl
    w = wl.CONFIGS[name]() if seed is None else wl.CONFIGS[name](seed=seed)
    if seed is not None:
        w = dataclasses.replace(w, name=f"{w.name}_seed{seed}")
    if layout != "combined":
        w = dataclasses.replace(w, layout=layout, name=f"{w.name}_{layout}")
    return w


def step_bytes(w, step, out_bytes=2):
    """Algorithmic bytes of decode ``step``: K/V of every view token read once, q read, out
    written, the appended tokens' K/V read and written."""
    T = w.view_tokens(step)                  # all problems, after this step's append
    kv = T * w.num_kv_heads * w.head_dim * 2 * 2
    q = w.num_problems * w.num_workers * w.num_q_heads * w.head_dim * 2
    out = w.num_problems * w.num_workers * w.num_q_heads * w.head_dim * out_bytes
    app = w.num_problems * w.num_workers * w.num_kv_heads * w.head_dim * 2 * 2 * 2
    return w.num_layers * (kv + q + out + app), w.num_layers * (kv + q)


# ---------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- oracle leg


def oracle_sample(w, seconds=12.0, max_steps=None):
    """Time the fp64 oracle (as it stands) on decode steps of ``w``: append + method form.
    Returns (seconds per step, steps timed, BLAS threads)."""
    from oracle import attention as A
    from oracle import run as orun
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    c = orun.prefill(w)
    times = []
    step = 0
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        orun.append_step(c, w, step)
        for layer in range(c.L):
            A.method(c, layer, orun.query(w, layer, step))
        c.step_end(__import__("workload").finished_mask(w, step))
        times.append(time.perf_counter() - t0)
        step += 1
        if time.perf_counter() - t_all > seconds or (max_steps and step >= max_steps):
            break
    return statistics.median(times), len(times), threads


def cpu_baseline(w, seconds=12.0):
    import workload as wl
    sample_w = wl.scaled(w, steps=64)
    per_step, n, threads = oracle_sample(sample_w, seconds)
    b, _ = step_bytes(w, 0)
    return {"value": b / per_step / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full decode steps of {w.name} (fp64 numpy method form: append, "
                      f"per-block query rotation, LSE merge), median {per_step * 1e3:.1f} ms/step"}


def slowest_rank_seconds(t, world, device=None):
    """The timed region's length on the slowest of the world's ranks (every rank gets it):
    one max all-reduce, the only collective of a timed run (replicas share no data)."""
    if world <= 1:
        return t
    import torch
    import torch.distributed as dist
    x = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def job_value(world, bytes_per_rank, t_slowest):
    """Whole-job GB/s: every rank streams the same workload; the job ends with its slowest rank."""
    return world * bytes_per_rank / t_slowest / 1e9


def workload_config(w):
    """The workload keys of a bench line's config (both arms)."""
    return {"workload": w.name, "layout": w.layout, "problems": w.num_problems,
            "workers": w.num_workers, "layers": w.num_layers, "H_q": w.num_q_heads,
            "H_kv": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
            "common_tokens": list(w.common_len)}


def run_reference(args):
    """The oracle (as it stands) on the host cores: W untimed decode steps, then exactly K timed
    ones, each a whole decode step of the same workload (append, method form, step end)."""
    import workload as wl
    from oracle import attention as A
    from oracle import run as orun
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    base = workload_for(args.config, args.layout, args.seed)
    w = wl.scaled(base, name=base.name, steps=args.warmup + args.steps + 1)
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    c = orun.prefill(w)

    def one_step(step):
        orun.append_step(c, w, step)
        for layer in range(c.L):
            A.method(c, layer, orun.query(w, layer, step))
        c.step_end(wl.finished_mask(w, step))

    for step in range(args.warmup):
        one_step(step)
    t0 = time.perf_counter()
    total = 0
    for step in range(args.warmup, args.warmup + args.steps):
        one_step(step)
        total += step_bytes(w, step)[0]
    t = time.perf_counter() - t0
    v = total / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "worker_tokens_per_s": w.num_problems * w.num_workers * args.steps / t,
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{args.steps} timed decode steps of {w.name} after "
                                       f"{args.warmup} untimed ones"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU leg


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import workload as wl
    from shared_kv_concurrent_gb300 import binding
    from shared_kv_concurrent_gb300.runner import WorkloadRunner, to_device_bf16

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    base = workload_for(args.config, args.layout, args.seed)
    e2e_steps = args.e2e_steps
    kv_mb = base.num_layers * base.view_tokens(0) * base.num_kv_heads * base.head_dim * 4 / 1e6
    layer_mb = kv_mb / base.num_layers                     # K/V of one layer of one cache
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if args.caches:
        R = args.caches
    elif (kv_mb - layer_mb) * 1e6 >= 2 * l2:
        R = 1          # one cache's other layers already stream more than 2x L2 per step
    else:
        R = max(4, int(math.ceil(2 * l2 / (kv_mb * 1e6))) + 1)
    per_cache = -(-(args.warmup + 2 * args.steps) // R) + 1
    w = wl.scaled(base, name=base.name, steps=per_cache + e2e_steps + 1)
    P, W, Hq, D, L = w.num_problems, w.num_workers, w.num_q_heads, w.head_dim, w.num_layers
    # R independent caches of the same workload, used in turn: consecutive steps touch
    # different K/V, and a cache comes back only after the other R-1 have streamed theirs, so
    # its K/V come from HBM without flushing L2 inside the timed region.
    # Between two reads of the same layer's K/V, everything else streams through L2.
    if (R * kv_mb - layer_mb) * 1e6 < 2 * l2:
        raise SystemExit(f"--caches {R}: the other {R * kv_mb - layer_mb:.0f} MB of K/V do not "
                         f"evict a layer from the {l2 / 1e6:.0f} MB L2; use more caches")
    runners = [WorkloadRunner(w, device=dev) for _ in range(R)]
    ctxs = [r.cache.ctx for r in runners]
    local = [0] * R                              # next decode step of each cache
    outs = [torch.empty(P, W, Hq, D, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    # Replace the lines the prefills left in L2 (written at normal priority, they would outlive
    # the kernel's evict-first K/V traffic and serve part of the last-built cache from L2).
    flush.zero_()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev).cuda_stream     # raw handle: no per-call lookup

    n_planned = [0]

    def plan_steps(n):
        """The next n steps, caches in turn: (cache, its step index, inputs resident in HBM)."""
        seq = []
        for _ in range(n):
            c = n_planned[0] % R
            n_planned[0] += 1
            seq.append((c, local[c]))
            local[c] += 1
        return [(c, st, runners[c].step_inputs(st)) for c, st in seq]

    def run_step(c, st, inp):
        runners[c].append(inp, stream=stream)
        runners[c].attend(inp, outs, stream=stream)
        runners[c].end(st, stream=stream)

    host_s = []
    for c, st, inp in plan_steps(args.warmup):
        t0 = time.perf_counter()
        run_step(c, st, inp)
        host_s.append(time.perf_counter() - t0)
        torch.cuda.synchronize()
    host_step = statistics.median(host_s)      # host time to submit one step (Python + C API)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    for ctx in ctxs:
        binding.hw_profile_read(ctx)                  # reset the launch counters
    timed = plan_steps(args.steps)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(uuid)
    time.sleep(0.3)
    # Submission runs ahead of the device: a bounded device-side delay first, long enough for the
    # host to enqueue every timed step, so that the events time the GPU's work and not the gaps
    # of a slower Python loop.  The host's own cost per step is reported beside
    # (host_us_per_step: the median over the timed steps' submissions, made while the device
    # sleeps) and is inside the e2e number.
    sm_hz = 2.07e9                             # GB300 maximum SM clock (cycles of the delay)

    def device_delay():
        # One SM spins while the host queues the steps (a kernel of torch's own: nothing here
        # may make the host wait for the device, or the steps would go out at host speed).
        torch.cuda._sleep(int(min(0.2, 3 * args.steps * host_step + 2e-3) * sm_hz))

    device_delay()
    e_start.record()
    total_bytes = 0
    submit_s = []                  # host time to submit each timed step (the device sleeps)
    for c, st, inp in timed:
        t0 = time.perf_counter()
        run_step(c, st, inp)
        submit_s.append(time.perf_counter() - t0)
        total_bytes += step_bytes(w, st)[0]
    e_end.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    launches = sum(int(binding.hw_profile_read(ctx)["launches"]) for ctx in ctxs)
    t_total = e_start.elapsed_time(e_end) / 1e3

    # Kernel timing pass: the same kind of steps again, now with the library recording CUDA
    # events directly around each attention kernel on its stream (kept out of the pass above
    # because an event between launches ends their programmatic chaining).
    for ctx in ctxs:
        binding.hw_profile_enable(ctx, True)
        binding.hw_profile_read(ctx)
    prof_steps = plan_steps(args.steps)
    attn_bytes = 0
    device_delay()
    for c, st, inp in prof_steps:
        run_step(c, st, inp)
        attn_bytes += step_bytes(w, st)[1]
    torch.cuda.synchronize()
    attn_ms_sum, attn_n, other_ms_sum = 0.0, 0, 0.0
    for ctx in ctxs:
        pr = binding.hw_profile_read(ctx)
        attn_ms_sum += pr["attention_ms"]
        attn_n += pr["timed_attention"]
        other_ms_sum += pr["merge_ms"] + pr["append_ms"]
        binding.hw_profile_enable(ctx, False)
    prof = {"attention_ms": attn_ms_sum, "timed_attention": attn_n,
            # the attention kernels' share of the library's kernel time in a step (events
            # around every kernel of the pass: attention, merge, append)
            "share": attn_ms_sum / max(1e-12, attn_ms_sum + other_ms_sum)}
    t_total = slowest_rank_seconds(t_total, world, dev)
    # End to end through the public API: inputs in pinned host memory.
    # (cache 0, L2 flushed before every step; one whole step at a time through
    # hw_decode_step_host: the packed K/V/Q copy in, append, attention, the output copy out,
    # step end and a stream synchronize)
    e2e = None
    if e2e_steps:
        runner = runners[0]
        first = local[0]
        host_in = [runner.packed_inputs(first + i) for i in range(e2e_steps)]
        host_out = torch.empty(L * P * W * Hq * D, dtype=torch.bfloat16).pin_memory()
        runner.cache.reserve_step_scratch(runner.n_step)
        e2e_times, e2e_bytes = [], 0
        for i in range(e2e_steps):
            s = first + i
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            runner.cache.decode_step_host(runner._n_step_ptr, host_in[i], host_out,
                                          runner.finished_for(s), sync=True, stream=stream)
            e2e_times.append(time.perf_counter() - t0)
            e2e_bytes += step_bytes(w, s)[0]
        h2d = host_in[0].numel()
        d2h = host_out.numel() * 2
        # (whole job, as `value`: every rank ran the same steps; the slowest rank's time)
        t_e2e = slowest_rank_seconds(sum(e2e_times), world, dev)
        e2e = {"value": job_value(world, e2e_bytes, t_e2e), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": 1e3 * t_e2e / e2e_steps, "steps": e2e_steps,
               "call": "hw_decode_step_host (one packed host-to-device copy, one copy back)"}

    for r in runners:
        st, info = r.cache.check_device_errors()
        if st != binding.HW_OK:
            raise RuntimeError(f"device error word set: {info}")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    value = job_value(world, total_bytes, t_total)
    # The attention kernel's time inside the timed chain: the chained step's device time (one
    # CUDA event pair around all timed steps), times the kernel's share of the step's kernel
    # time from the pass with events around every kernel, per attention launch (one per layer
    # per step).  That pass's own per-launch figure, unchained (each launch pays its full
    # start-up), is reported beside it.
    attn_launch_bytes = attn_bytes / max(1, prof["timed_attention"])   # one launch per layer
    attn_ms_isolated = prof["attention_ms"] / max(1, prof["timed_attention"])
    ncu_share = captured_share() if w.name == "w8_common32768_paged" else None
    share = ncu_share if ncu_share is not None else prof["share"]
    attn_ms = 1e3 * t_total * share / (args.steps * L)
    achieved = attn_launch_bytes / (attn_ms / 1e3) / 1e9
    achieved_isolated = attn_launch_bytes / (attn_ms_isolated / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {**workload_config(w), "view_tokens_first_timed_step":
                   w.view_tokens(timed[0][1]), "parallelism": f"replicas{world}",
                   "l2": (f"inputs larger than L2: {R} independent cache(s) of this workload "
                          f"({kv_mb:.0f} MB of K/V each) used in turn, so a layer's K/V return "
                          f"only after {R * kv_mb - layer_mb:.0f} MB of other K/V; no flush in "
                          f"the timed region; the e2e leg flushes L2 (2x L2 memset) before "
                          f"every step"),
                   "timing": "one CUDA event pair around all timed steps",
                   "delay": ("before the start event one SM spins while the host queues the "
                             "timed steps"),
                   "step": "append 1 token/worker + concurrent attention + step end"},
        "pct_of_peak": 100.0 * value / world / peak,
        "worker_tokens_per_s": world * P * W * args.steps / t_total,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": captured_traffic() if w.name == "w8_common32768_paged" else None,
                     "peak_kind": peak_kind,
                     "kernel": "concurrent attention (split-K partials)",
                     "kernel_ms": attn_ms,
                     "kernel_timing": "in the timed chain: ms_per_step per layer x the kernel's "
                                      "share of the step's kernel time"
                                      + (" (committed ncu launch list of these kernel sources)"
                                         if ncu_share is not None else
                                         " (events around each kernel in a second pass)"),
                     "share_of_step": share,
                     "share_of_step_events": prof["share"],
                     "isolated": {"kernel_ms": attn_ms_isolated, "achieved": achieved_isolated,
                                  "frac": achieved_isolated / peak,
                                  "timing": "events directly around each launch, no chaining"},
                     "algorithmic_bytes_per_launch": attn_launch_bytes},
        "gpu_launches": launches,
        "host_us_per_step": 1e6 * statistics.median(submit_s),
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(base, seconds=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c4")
    ap.add_argument("--layout", default="combined",
                    choices=["combined", "step_wise", "contiguous", "no_sync"],
                    help="cache layout of the workload (the default is the method's own)")
    ap.add_argument("--seed", type=int, default=None,
                    help="another master seed for the workload (block lengths, page order, "
                         "tensors); the default is the workload's own")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--caches", type=int, default=0,
                    help="independent caches of the workload used in turn (0: enough that the "
                         "K/V read between two reads of a layer exceed 2x L2; 4 or more when "
                         "one cache is smaller than that)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.caches < 0:
        ap.error("--caches must be 0 (automatic) or positive")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
