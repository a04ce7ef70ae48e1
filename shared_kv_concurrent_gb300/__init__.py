"""GB300-native concurrent attention for Hogwild! Inference.

The computation lives in ``libhogwild.so`` (C ABI: ``include/hogwild.h``; CUDA kernels for
sm_103a under ``csrc/``).  ``binding`` is a thin ctypes layer with the same names as the C
entry points; ``HogwildCache`` below only owns the device buffers (allocated with torch) and
forwards every call to the library.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import binding
from .binding import (HW_OUT_BF16, HW_OUT_F32, HogwildError, hw_config)

__all__ = ["HogwildCache", "HogwildError", "LAYOUTS", "binding", "config_for"]


LAYOUTS = {"combined": 0, "step_wise": 1, "contiguous": 2, "no_sync": 3}   # HW_LAYOUT_*


def config_for(*, num_problems, num_workers, num_layers, num_q_heads, num_kv_heads, head_dim,
               page_size, num_pages, max_position, rope_theta, contiguous=False,
               max_segments=0, max_append_tokens=0, layout="combined") -> hw_config:
    return hw_config(num_problems, num_workers, num_layers, num_q_heads, num_kv_heads, head_dim,
                     page_size, int(bool(contiguous)), num_pages, max_position, max_segments,
                     max_append_tokens, float(rope_theta), LAYOUTS[layout], 0)


class HogwildCache:
    """One library context plus the torch-owned pools and workspace it runs on."""

    def __init__(self, cfg: hw_config, page_order=None, device="cuda"):
        import torch
        self.cfg = cfg
        self.device = torch.device(device)
        pool_bytes = binding.hw_pool_size(cfg)
        ws_bytes = binding.hw_workspace_size(cfg)
        self.k_pool = torch.empty(pool_bytes // 2, dtype=torch.bfloat16, device=self.device)
        self.v_pool = torch.empty(pool_bytes // 2, dtype=torch.bfloat16, device=self.device)
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        self.ctx = binding.hw_create(cfg, self.k_pool, self.v_pool, self.workspace, page_order)

    @classmethod
    def from_workload(cls, w, max_segments: int = 0, device="cuda") -> "HogwildCache":
        cfg = config_for(num_problems=w.num_problems, num_workers=w.num_workers,
                         num_layers=w.num_layers, num_q_heads=w.num_q_heads,
                         num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                         page_size=w.page_size, num_pages=w.num_pages(),
                         max_position=w.max_position(), rope_theta=w.rope_theta,
                         contiguous=w.contiguous, max_segments=max_segments,
                         layout=getattr(w, "layout", "combined"))
        return cls(cfg, page_order=w.page_order(), device=device)

    # -- the step protocol ---------------------------------------------------------------

    def append_kv(self, layer: int, n_new, k_raw, v_raw, stream=None) -> None:
        binding.hw_append_kv(self.ctx, layer, n_new, k_raw, v_raw, stream)

    def compact_segments(self, problem: int, first: int, count: int, stream=None) -> None:
        """Merge common segments first .. first+count-1 into one RoPE frame (between steps)."""
        binding.hw_compact_segments(self.ctx, problem, first, count, stream)

    def compact_auto(self, max_paragraphs: int, stream=None) -> int:
        """Merge the committed paragraphs of problems that have more than max_paragraphs
        (hw_compact_auto); returns the number of merges."""
        return binding.hw_compact_auto(self.ctx, max_paragraphs, stream)

    def concurrent_attention_mq(self, layer: int, q, n_q, out=None, out_dtype: str = "bf16",
                                lse=None, stream=None):
        """Several causal query tokens per worker (the last n_q[p][w] tokens of its block)."""
        import torch
        dt = HW_OUT_F32 if out_dtype == "f32" else HW_OUT_BF16
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32 if dt == HW_OUT_F32 else torch.bfloat16,
                              device=q.device)
        binding.hw_concurrent_attention_mq(self.ctx, layer, q, n_q, out, dt, lse, stream)
        return out

    def concurrent_attention(self, layer: int, q, out=None, out_dtype: str = "bf16", lse=None,
                             stream=None):
        import torch
        dt = HW_OUT_F32 if out_dtype == "f32" else HW_OUT_BF16
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32 if dt == HW_OUT_F32 else torch.bfloat16,
                              device=q.device)
        binding.hw_concurrent_attention(self.ctx, layer, q, out, dt, lse, stream)
        return out

    def concurrent_attention_range(self, layer: int, q, ranges, out=None, lse=None, stream=None):
        """Attention over entries [ranges[p][0], ranges[p][1]) of each problem (segment order):
        returns (out fp32, lse fp32), normalised over the selected keys."""
        import torch
        P, W, Hq = q.shape[0], q.shape[1], q.shape[2]
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((P, W, Hq), dtype=torch.float32, device=q.device)
        binding.hw_concurrent_attention_range(self.ctx, layer, q, ranges, out, lse, stream)
        return out, lse

    def entry_totals(self):
        """Entries of every problem in segment order (common segments, then the workers'
        blocks), this step's appended tokens included: the extent hw_concurrent_attention_range
        numbers."""
        totals = []
        for p in range(self.cfg.num_problems):
            common, live = binding.hw_get_blocks(self.ctx, p, self.cfg.num_workers)
            n = 0
            for sid in common + live:
                _, _, length, pending, _ = binding.hw_get_segment(self.ctx, sid)
                n += length + pending
            totals.append(n)
        return totals

    def step_end(self, finished=None, stream=None) -> None:
        binding.hw_step_end(self.ctx, finished, stream)

    def decode_step_host(self, n_new, in_host, out_host, finished=None, out_dtype: str = "bf16",
                         sync: bool = True, stream=None) -> None:
        """One decode step from host memory (hw_decode_step_host): ``in_host`` a page-locked
        uint8 CPU tensor holding the packed [K][V][Q] input, ``out_host`` a page-locked CPU
        tensor of L*P*W*H_q*D elements of out_dtype.  The device scratch is kept between calls
        (grown when a step needs more)."""
        dt = HW_OUT_F32 if out_dtype == "f32" else HW_OUT_BF16
        scratch = getattr(self, "_step_scratch", None)
        if scratch is None:
            scratch = self.reserve_step_scratch(n_new, out_dtype)
        args = (in_host.data_ptr(), in_host.numel() * in_host.element_size(), out_host.data_ptr(),
                dt, finished)
        try:
            binding.hw_decode_step_host(self.ctx, n_new, *args, scratch.data_ptr(),
                                        scratch.numel(), sync, stream)
        except HogwildError as e:
            # A scratch too small is refused before anything is enqueued: grow it and retry.
            # (The size is asked for only then, not on every step.)
            if (e.status != binding.HW_ERR_CAPACITY or
                    binding.hw_step_scratch_size(self.ctx, n_new, dt) <= scratch.numel()):
                raise
            scratch = self.reserve_step_scratch(n_new, out_dtype)
            binding.hw_decode_step_host(self.ctx, n_new, *args, scratch.data_ptr(),
                                        scratch.numel(), sync, stream)

    def reserve_step_scratch(self, n_new, out_dtype: str = "bf16"):
        """The device scratch of decode_step_host for the counts n_new, allocated (or grown)
        now rather than inside the first step."""
        import torch
        dt = HW_OUT_F32 if out_dtype == "f32" else HW_OUT_BF16
        need = binding.hw_step_scratch_size(self.ctx, n_new, dt)
        scratch = getattr(self, "_step_scratch", None)
        if scratch is None or scratch.numel() < need:
            # (a larger buffer may only replace the old one once no step still uses it)
            torch.cuda.synchronize(self.device)
            scratch = self._step_scratch = torch.empty(need, dtype=torch.uint8, device=self.device)
        return scratch

    def check_device_errors(self, stream=None):
        return binding.hw_check_device_errors(self.ctx, stream)

    # -- read-back ----------------------------------------------------------------------

    def tables(self) -> dict:
        nseg, free = binding.hw_get_counts(self.ctx)
        segs = [tuple(binding.hw_get_segment(self.ctx, s)) for s in range(nseg)]
        common, live = [], []
        for p in range(self.cfg.num_problems):
            c, l = binding.hw_get_blocks(self.ctx, p, self.cfg.num_workers)
            common.append(c)
            live.append(l)
        return {"segments": [(a, b, c, d, list(e)) for a, b, c, d, e in segs],
                "common": common, "live": live, "free_count": free}

    def view(self, p: int, w: int):
        return binding.hw_get_view(self.ctx, p, w)

    def pools(self, layer: int):
        """K and V pools of one layer as [num_pages][H_kv][S][D] bf16 tensors (views)."""
        c = self.cfg
        n = c.num_pages * c.num_kv_heads * c.page_size * c.head_dim
        shape = (c.num_pages, c.num_kv_heads, c.page_size, c.head_dim)
        return (self.k_pool[layer * n:(layer + 1) * n].view(shape),
                self.v_pool[layer * n:(layer + 1) * n].view(shape))

    def close(self) -> None:
        if getattr(self, "ctx", None):
            binding.hw_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
