"""Drive the oracle cache through a seeded workload (test infrastructure only).

Prefill: every layer appends the whole common block and every worker's block, then the step
ends with no commit.  Decode step t: every layer appends one new token per worker, attention
runs, then the step ends and the workload's commits (if any) are applied -- the order of the
Hogwild! inference flow (gentlecold.top summary, section 8).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

import workload as wl

from .cache import HogwildCache


def bf16(bits: np.ndarray) -> np.ndarray:
    return wl.bf16_bits_to_f32(bits)


def new_cache(w: wl.Workload, layers: Optional[int] = None) -> HogwildCache:
    return HogwildCache(w.num_problems, w.num_workers, layers or w.num_layers, w.num_kv_heads,
                        w.head_dim, w.rope_theta, w.page_size, w.num_pages(),
                        contiguous=w.contiguous, page_order=w.page_order(), layout=w.layout)


def prefill(w: wl.Workload, layers: Optional[int] = None,
            layer_ids: Optional[Sequence[int]] = None) -> HogwildCache:
    """Cache holding the workload's pre-step blocks (layer l uses the layer-l draws).

    ``layer_ids``: keep only these workload layers (cache layer i holds workload layer
    layer_ids[i]) -- the tables do not depend on the layer, so a few layers pin a deep model."""
    ids = list(layer_ids) if layer_ids is not None else list(range(layers or w.num_layers))
    c = new_cache(w, len(ids))
    n = wl.prefill_block_lengths(w)
    for i, layer in enumerate(ids):
        k, v = wl.prefill_kv(w, layer)
        c.append(i, n, bf16(k), bf16(v))
    c.step_end(np.zeros((w.num_problems, w.num_workers), np.uint8))
    return c


def append_step(c: HogwildCache, w: wl.Workload, step: int,
                layer_ids: Optional[Sequence[int]] = None) -> None:
    n = wl.step_n_new(w)
    ids = list(layer_ids) if layer_ids is not None else list(range(c.L))
    for i, layer in enumerate(ids):
        k, v = wl.step_kv(w, layer, step)
        c.append(i, n, bf16(k), bf16(v))


def query(w: wl.Workload, layer: int, step: int) -> np.ndarray:
    return bf16(wl.step_q(w, layer, step)).astype(np.float64)
