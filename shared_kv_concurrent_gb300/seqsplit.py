"""Sequence split of a decode step over several GPUs.

Hogwild! Inference (summary at gentlecold.top, section 9) splits the attention work over KV
entries and reduces the partial results afterwards.  Across GPUs that becomes: every rank
holds the same cache tables, attends over its own range of every problem's entries with
``hw_concurrent_attention_range`` (normalised output and log-sum-exp per query row), the
ranks all-gather those parts -- one collective for the outputs and one for the log-sum-exps,
plain ring all-gathers (NCCL on GPUs, gloo on CPU), no multicast -- and each rank merges them
with ``hw_merge_attention``.  The entries are numbered in segment order (common segments in
commit order, then the workers' blocks by id); ``split_entries`` cuts them into contiguous
ranges of nearly equal size, one per rank.

Only the exchange lives here; every step of the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def split_entries(totals: Sequence[int], world: int) -> np.ndarray:
    """Contiguous ranges [begin, end) of every problem's entries, one per rank: int64
    [world][P][2]; rank r gets entries floor(r * n / world) .. floor((r + 1) * n / world)."""
    if world < 1:
        raise ValueError("world must be at least 1")
    n = np.asarray(totals, dtype=np.int64)
    r = np.arange(world + 1, dtype=np.int64)[:, None]
    edges = (r * n[None, :]) // world                     # [world + 1][P]
    return np.stack([edges[:-1], edges[1:]], axis=-1)


def gather_parts(out, lse, group=None):
    """All-gather of every rank's part: out [...][D] and lse [...] (the same shapes on every
    rank) -> parts_out [world][...][D], parts_lse [world][...], in rank order."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts_out = torch.empty((world,) + tuple(out.shape), dtype=out.dtype, device=out.device)
    parts_lse = torch.empty((world,) + tuple(lse.shape), dtype=lse.dtype, device=lse.device)
    dist.all_gather(list(parts_out.unbind(0)), out.contiguous(), group=group)
    dist.all_gather(list(parts_lse.unbind(0)), lse.contiguous(), group=group)
    return parts_out, parts_lse


def merge_parts(parts_out, parts_lse, out, out_dtype: str = "bf16", lse=None, stream=None):
    """The library's log-sum-exp merge of gathered parts into out (and lse)."""
    from . import binding
    dt = binding.HW_OUT_F32 if out_dtype == "f32" else binding.HW_OUT_BF16
    binding.hw_merge_attention(parts_out, parts_lse, out, dt, lse, stream)
    return out
