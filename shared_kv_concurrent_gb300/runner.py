"""Drive the library through a seeded synthetic workload (device side).

Prefill appends every block of every layer, then ends the step with no commit.  A decode step
appends one token per worker to every layer, runs the concurrent attention of every layer and
ends the step with the workload's commits -- the order of the Hogwild! inference flow (append,
attend, commit at step end).
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np

import workload as wl

from . import HogwildCache


def to_device_bf16(bits: np.ndarray, device="cuda"):
    """uint16 bf16 bit patterns -> torch bf16 tensor on ``device`` (exact)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


class WorkloadRunner:
    def __init__(self, w: wl.Workload, device="cuda", max_segments: int = 0):
        self.w = w
        self.device = device
        self.cache = HogwildCache.from_workload(w, max_segments=max_segments, device=device)
        n = wl.prefill_block_lengths(w)
        keep = []          # k/v stay alive until the step end has written them (hw_append_kv)
        for layer in range(w.num_layers):
            k, v = wl.prefill_kv(w, layer)
            if k.shape[0] == 0:
                self.cache.append_kv(layer, n, None, None)
                continue
            kd, vd = to_device_bf16(k, device), to_device_bf16(v, device)
            self.cache.append_kv(layer, n, kd, vd)
            keep.append((kd, vd))
        self.cache.step_end(np.zeros((w.num_problems, w.num_workers), np.uint8))
        del keep
        self.n_step = np.ascontiguousarray(wl.step_n_new(w), dtype=np.int32)
        self._n_step_ptr = self.n_step.ctypes.data          # (the arrays live with the runner)
        self._no_commit = np.zeros((w.num_problems, w.num_workers), np.uint8)
        self._no_commit_ptr = self._no_commit.ctypes.data

    def step_inputs(self, step: int):
        """Device tensors (k[L], v[L], q[L]) of decode ``step``."""
        ks, vs, qs = [], [], []
        for layer in range(self.w.num_layers):
            k, v = wl.step_kv(self.w, layer, step)
            ks.append(to_device_bf16(k, self.device))
            vs.append(to_device_bf16(v, self.device))
            qs.append(to_device_bf16(wl.step_q(self.w, layer, step), self.device))
        return ks, vs, qs

    def append(self, inputs, stream=None) -> None:
        """``stream``: a torch stream or raw cudaStream_t handle; None = torch's current one."""
        ks, vs, _ = inputs
        for layer in range(self.w.num_layers):
            self.cache.append_kv(layer, self._n_step_ptr, ks[layer], vs[layer], stream)

    def attend(self, inputs, outs: List, lses: Optional[List] = None, out_dtype="bf16",
               stream=None) -> None:
        _, _, qs = inputs
        for layer in range(self.w.num_layers):
            self.cache.concurrent_attention(layer, qs[layer], outs[layer], out_dtype,
                                            None if lses is None else lses[layer], stream)

    def finished_for(self, step: int):
        """The workload's commit mask after ``step`` (the address of a zero mask if none)."""
        return wl.finished_mask(self.w, step) if step in self.w.commit_steps else self._no_commit_ptr

    def packed_inputs(self, step: int):
        """Page-locked uint8 CPU tensor [K(L)][V(L)][Q(L)] of decode ``step``: the input of
        hw_decode_step_host."""
        import torch
        parts_k, parts_v, parts_q = [], [], []
        for layer in range(self.w.num_layers):
            k, v = wl.step_kv(self.w, layer, step)
            parts_k.append(np.ascontiguousarray(k).ravel())
            parts_v.append(np.ascontiguousarray(v).ravel())
            parts_q.append(np.ascontiguousarray(wl.step_q(self.w, layer, step)).ravel())
        flat = np.concatenate(parts_k + parts_v + parts_q).astype(np.uint16).view(np.uint8)
        return torch.from_numpy(flat.copy()).pin_memory()

    def end(self, step: int, finished=None, stream=None) -> None:
        if finished is None:
            finished = self.finished_for(step)
        self.cache.step_end(finished, stream)
