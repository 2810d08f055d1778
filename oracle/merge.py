"""Oracle: combining attention results over disjoint key sets by log-sum-exp.

Test infrastructure only (see the package docstring).

Source: [AK] section four ("How the FlashAttention cascade merges results"):
each part is already normalised, so the parts are weighted by their
unnormalised mass Z_k, O = (sum Z_k O_k) / (sum Z_k); the worked example has
Z = 3, 1 and O = 2, 10, giving 4 (not the plain mean 6). With base-2
log-sum-exps l_k (Z_k = 2^l_k): O = sum 2^l_k O_k / sum 2^l_k and
l = log2 sum 2^l_k.
"""
from __future__ import annotations

import numpy as np


def merge_states(outs, lse2s):
    """outs: [K][..., d], lse2s: [K][...] (base 2). Parts with lse2 = -inf carry no mass."""
    outs = np.asarray(outs, dtype=np.float64)
    l = np.asarray(lse2s, dtype=np.float64)
    top = l.max(axis=0)                   # factor 2^top out of every Z_k
    z = np.exp2(l - top)
    Z = z.sum(axis=0)
    o = (z[..., None] * outs).sum(axis=0) / Z[..., None]
    return o, top + np.log2(Z)
