"""Seeded synthetic workloads for the Hogwild! concurrent-attention decode step.

This module only says WHAT the inputs are: the shapes of each benchmark configuration, the
seeded block lengths and physical page permutation, and seeded N(0,1) query/key/value draws
rounded to bf16.  It performs none of the method's arithmetic (no RoPE, no attention, no cache
bookkeeping), so that the fp64 CPU oracle and the CUDA library can both consume it without
sharing any code that computes a result.

Draw protocol.  Every tensor comes from its own counter-keyed stream
``PCG64(SeedSequence([seed, TAG_TENSOR, layer, phase, problem, block, tensor_id]))``: one
master seed per configuration and a per-unit key, in the spirit of deriving per-unit seeds from
one master seed.  ``phase`` is 0 for the cache prefill and ``t + 1`` for decode step ``t``;
``block`` is 0 for the common block and ``1 + w`` for worker ``w``; ``tensor_id`` is 0 (K),
1 (V) or 2 (Q).  Values are drawn as float32 N(0,1) and rounded to bf16 with
round-to-nearest-even; both sides consume exactly those bf16 values.

The shapes follow the workloads of Hogwild! Inference (gentlecold.top summary, section 9: a
common block plus one current block per worker, all layers sharing block lengths), with sizes
chosen for one GB300; the models and datasets of the paper are not used.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import numpy as np

TAG_LENGTHS = 1
TAG_PAGES = 2
TAG_TENSOR = 3
TAG_FINISHED = 4

K_ID, V_ID, Q_ID = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic Hogwild! problem set.

    ``common_len[p]`` and ``worker_len[p][w]`` are the block lengths BEFORE the first timed
    step; every decode step appends one token per worker and then attends.
    """

    name: str
    num_problems: int
    num_workers: int
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    rope_theta: float
    page_size: int          # tokens per page; for a contiguous cache, the block capacity
    contiguous: bool        # True: each block is one [H_kv][cap][D] region
    random_page_order: bool
    seed: int
    common_len: Tuple[int, ...]
    worker_len: Tuple[Tuple[int, ...], ...]
    steps: int = 1          # decode steps the workload runs
    commit_steps: Tuple[int, ...] = ()  # steps after which every worker commits its block
    layout: str = "combined"            # cache layout: combined, step_wise, contiguous, no_sync

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def rows_per_kv_head(self) -> int:
        return self.num_workers * self.group

    def view_tokens(self, step: int = 0) -> int:
        """Tokens every worker sees at ``step`` (after that step's append), all problems."""
        return sum(self.common_len) + sum(sum(r) for r in self.worker_len) + \
            (step + 1) * self.num_workers * self.num_problems

    def max_position(self) -> int:
        """Upper bound on any view length over the workload's steps (RoPE table rows)."""
        per_problem = [self.common_len[p] + sum(self.worker_len[p]) +
                       (self.steps + 1) * self.num_workers for p in range(self.num_problems)]
        return max(per_problem) + 1

    def num_pages(self) -> int:
        """Pages per layer that the workload can consume, with slack."""
        S = self.page_size
        if self.contiguous:
            # one page per block, plus one per commit (a fresh block per committed worker)
            return self.num_problems * (1 + self.num_workers) * (1 + len(self.commit_steps)) + 4
        total = 0
        extra = self.steps + 1
        for p in range(self.num_problems):
            total += -(-self.common_len[p] // S)
            for w in range(self.num_workers):
                total += -(-(self.worker_len[p][w] + extra) // S)
        # a commit starts a fresh block per worker: at most one partial page each
        total += self.num_problems * self.num_workers * (len(self.commit_steps) + 1)
        return total + 8

    def page_order(self) -> np.ndarray:
        """Initial free-list order of physical pages (int32)."""
        n = self.num_pages()
        if not self.random_page_order:
            return np.arange(n, dtype=np.int32)
        g = _rng(self.seed, TAG_PAGES)
        return g.permutation(n).astype(np.int32)


def _rng(seed: int, *keys: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed)] + [int(k) for k in keys])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits.

    Inputs here are finite normal draws, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def draw_bf16(w: Workload, layer: int, phase: int, problem: int, block: int, tensor_id: int,
              shape: Sequence[int]) -> np.ndarray:
    """Seeded N(0,1) tensor rounded to bf16, returned as uint16 bits of ``shape``."""
    g = _rng(w.seed, TAG_TENSOR, layer, phase, problem, block, tensor_id)
    x = g.standard_normal(size=tuple(shape), dtype=np.float32)
    return f32_to_bf16_bits(x)


def prefill_block_lengths(w: Workload) -> np.ndarray:
    """n_new table [P][W+1] of the cache prefill (index 0 = common, 1 + w = worker w)."""
    n = np.zeros((w.num_problems, w.num_workers + 1), dtype=np.int32)
    for p in range(w.num_problems):
        n[p, 0] = w.common_len[p]
        for k in range(w.num_workers):
            n[p, 1 + k] = w.worker_len[p][k]
    return n


def prefill_kv(w: Workload, layer: int) -> Tuple[np.ndarray, np.ndarray]:
    """Raw (unrotated) K and V of the prefill, bf16 bits [sum n][H_kv][D].

    Token order: problem-major, then block 0 (common), 1..W (workers), each in position order.
    """
    ks, vs = [], []
    for p in range(w.num_problems):
        lens = [w.common_len[p]] + list(w.worker_len[p])
        for b, n in enumerate(lens):
            if n == 0:
                continue
            ks.append(draw_bf16(w, layer, 0, p, b, K_ID, (n, w.num_kv_heads, w.head_dim)))
            vs.append(draw_bf16(w, layer, 0, p, b, V_ID, (n, w.num_kv_heads, w.head_dim)))
    if not ks:
        z = np.zeros((0, w.num_kv_heads, w.head_dim), dtype=np.uint16)
        return z, z.copy()
    return np.concatenate(ks), np.concatenate(vs)


def step_n_new(w: Workload) -> np.ndarray:
    """n_new table of one decode step: one token per worker, none for the common block."""
    n = np.zeros((w.num_problems, w.num_workers + 1), dtype=np.int32)
    n[:, 1:] = 1
    return n


def step_kv(w: Workload, layer: int, step: int) -> Tuple[np.ndarray, np.ndarray]:
    """New raw K and V of decode ``step`` (one token per worker), bf16 bits [P*W][H_kv][D]."""
    ks, vs = [], []
    for p in range(w.num_problems):
        for k in range(w.num_workers):
            ks.append(draw_bf16(w, layer, step + 1, p, 1 + k, K_ID, (1, w.num_kv_heads, w.head_dim)))
            vs.append(draw_bf16(w, layer, step + 1, p, 1 + k, V_ID, (1, w.num_kv_heads, w.head_dim)))
    return np.concatenate(ks), np.concatenate(vs)


def step_q(w: Workload, layer: int, step: int) -> np.ndarray:
    """Unrotated queries of decode ``step``, bf16 bits [P][W][H_q][D]."""
    q = np.empty((w.num_problems, w.num_workers, w.num_q_heads, w.head_dim), dtype=np.uint16)
    for p in range(w.num_problems):
        for k in range(w.num_workers):
            q[p, k] = draw_bf16(w, layer, step + 1, p, 1 + k, Q_ID, (w.num_q_heads, w.head_dim))
    return q


def finished_mask(w: Workload, step: int, bernoulli: Optional[float] = None) -> np.ndarray:
    """Which workers end their paragraph after decode ``step`` ([P][W] uint8).

    By default every worker commits after the steps in ``commit_steps``; with ``bernoulli``
    each worker commits independently with that probability (seeded per step).
    """
    m = np.zeros((w.num_problems, w.num_workers), dtype=np.uint8)
    if bernoulli is not None:
        g = _rng(w.seed, TAG_FINISHED, step)
        m[:] = (g.random((w.num_problems, w.num_workers)) < bernoulli).astype(np.uint8)
    elif step in w.commit_steps:
        m[:] = 1
    return m


# --------------------------------------------------------------------------------------------
# The benchmark configurations.  Index 0 is the small case the oracle finishes in seconds.


def _uniform_lengths(seed: int, P: int, W: int, lo: int, hi: int, stream: int = 0):
    g = _rng(seed, TAG_LENGTHS, stream)
    return tuple(tuple(int(x) for x in g.integers(lo, hi + 1, size=W)) for _ in range(P))


def tiny(contiguous: bool = False, seed: int = 1000) -> Workload:
    """W=2, H_q 8, H_kv 2, D 64, theta 1e4; common 512, each worker block 64; views C+B+A / C+A+B."""
    return Workload(name="tiny_w2_c512" + ("_contig" if contiguous else ""), num_problems=1,
                    num_workers=2, num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=64,
                    rope_theta=1e4, page_size=(640 if contiguous else 256), contiguous=contiguous,
                    random_page_order=False, seed=seed, common_len=(512,),
                    worker_len=((64, 64),), steps=4)


def c2(seed: int = 1001) -> Workload:
    """W=2, H_q 40, H_kv 8, D 128, theta 1e6; common 4096, worker blocks 256; contiguous cache."""
    return Workload(name="w2_common4096_contig", num_problems=1, num_workers=2, num_layers=1,
                    num_q_heads=40, num_kv_heads=8, head_dim=128, rope_theta=1e6,
                    page_size=4224, contiguous=True, random_page_order=False, seed=seed,
                    common_len=(4096,), worker_len=((256, 256),), steps=64)


def c3(seed: int = 1002) -> Workload:
    """W=4, H_q 64, H_kv 8, D 128; common 16384, worker blocks U[0,1024]; 64 layers."""
    return Workload(name="w4_common16384_64layers", num_problems=1, num_workers=4, num_layers=64,
                    num_q_heads=64, num_kv_heads=8, head_dim=128, rope_theta=1e6,
                    page_size=256, contiguous=False, random_page_order=False, seed=seed,
                    common_len=(16384,), worker_len=_uniform_lengths(seed, 1, 4, 0, 1024),
                    steps=16)


def c4(seed: int = 1003) -> Workload:
    """W=8, H_q 64, H_kv 8, D 128; common 32768 + worker blocks U[128,2048]; paged, permuted."""
    return Workload(name="w8_common32768_paged", num_problems=1, num_workers=8, num_layers=1,
                    num_q_heads=64, num_kv_heads=8, head_dim=128, rope_theta=1e6,
                    page_size=256, contiguous=False, random_page_order=True, seed=seed,
                    common_len=(32768,), worker_len=_uniform_lengths(seed, 1, 8, 128, 2048),
                    steps=400)


def c5(seed: int = 1004) -> Workload:
    """16 problems x W=4, H_q 32, H_kv 8, D 128; lognormal common lengths; 200 steps."""
    g = _rng(seed, TAG_LENGTHS, 1)
    common = np.clip(np.round(g.lognormal(mean=math.log(8192.0), sigma=0.7, size=16)),
                     1024, 65536).astype(int)
    return Workload(name="p16_w4_lognormal_200steps", num_problems=16, num_workers=4,
                    num_layers=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    rope_theta=1e6, page_size=256, contiguous=False, random_page_order=False,
                    seed=seed, common_len=tuple(int(c) for c in common),
                    worker_len=_uniform_lengths(seed, 16, 4, 0, 512), steps=200,
                    commit_steps=(63, 127, 191))


CONFIGS = {"tiny": tiny, "c2": c2, "c3": c3, "c4": c4, "c5": c5}


def scaled(w: Workload, *, name: Optional[str] = None, common_len=None, worker_len=None,
           num_layers=None, steps=None, num_problems=None, commit_steps=None) -> Workload:
    """A smaller copy of a workload (same heads, dims, seed protocol) for quick parity runs."""
    kw = {}
    if num_problems is not None:
        kw["num_problems"] = num_problems
    if common_len is not None:
        kw["common_len"] = tuple(common_len)
    if worker_len is not None:
        kw["worker_len"] = tuple(tuple(r) for r in worker_len)
    if num_layers is not None:
        kw["num_layers"] = num_layers
    if steps is not None:
        kw["steps"] = steps
    if commit_steps is not None:
        kw["commit_steps"] = tuple(commit_steps)
    kw["name"] = name or (w.name + "_scaled")
    return dataclasses.replace(w, **kw)
