"""Rotary position embedding in fp64 (oracle; test infrastructure only).

rho(x, p) rotates each pair (x_i, x_{i+D/2}) by the angle p * f_i with f_i = theta^(-2i/D),
i < D/2 ("half-split" pairing).  The Hogwild! summary (gentlecold.top, section 5) writes the
attention score as rho(q, i_q) . rho(k, i_k) and relies only on its dependence on i_q - i_k; it
does not fix the pairing, so this oracle takes the half-split pairing of the Qwen-family models
the paper evaluates.  Every identity the method uses holds for either pairing.
"""
from __future__ import annotations

import numpy as np


def inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """f_i = theta^(-2i/D) for i = 0 .. D/2-1, fp64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """rho(x, pos) in fp64.

    ``x`` has shape [..., D]; ``pos`` is a scalar or an array broadcastable to ``x.shape[:-1]``
    (positions may be any integers, including negative ones).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    out = np.empty(np.broadcast_shapes(x.shape, c.shape[:-1] + (D,)), dtype=np.float64)
    out[..., :h] = x1 * c - x2 * s
    out[..., h:] = x2 * c + x1 * s
    return out
