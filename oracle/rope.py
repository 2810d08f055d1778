"""Oracle: rotary position embedding in fp64.

Test infrastructure only (see the package docstring).

The pages fix only where RoPE is applied: node i is rotated at position
vc + depth[i] ([TS] "Position follows depth, slot follows node index"; [AK]
section two). They do not print the rotation itself; the reading taken is the
Llama rotate-half form: pairs (x_k, x_{k+d/2}) for k < d/2 rotate by angle
pos * theta^(-2k/d).
"""
from __future__ import annotations

import numpy as np


def inv_freq(d: int, theta: float) -> np.ndarray:
    k = np.arange(d // 2, dtype=np.float64)
    return float(theta) ** (-2.0 * k / d)


def rotate(x, pos, theta: float) -> np.ndarray:
    """x: [..., d] (any float), pos: scalar or array broadcastable to x[..., 0]."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
