"""Oracle: the target's argmax at every verify row, and the walk fed by it.

Test infrastructure only (see the package docstring).

Sources:
* [MI] "Walking the accepted path": target_predict is the target's argmax at
  each node's position, computed for all nodes by the single verify forward;
  the walk compares draft tokens against it.
* [MI] the worked (steps, topk, nodes) = (5, 4, 8) iteration, step 5:
  eagle_sample takes the argmax over all 8 rows, then calls the greedy walk.

Readings taken (the pages state no tie or NaN rule): among equal maxima the
lowest vocabulary index wins; a NaN counts as larger than every number, so
the first NaN of a row wins; -0.0 and +0.0 are equal. These are NumPy's
argmax rules, and the logits are compared as given (fp32), never rounded.
"""
from __future__ import annotations

import numpy as np

from . import walk as _walk


def row_argmax(logits):
    """logits [rows][vocab] -> int32 [rows]: the argmax of each row."""
    x = np.asarray(logits)
    if x.ndim != 2 or x.shape[1] < 1:
        raise ValueError("logits must be [rows][vocab] with vocab >= 1")
    return np.argmax(x, axis=1).astype(np.int32)


def greedy_walk_from_logits(parents, draft_tokens, logits):
    """[B][N] trees and draft tokens, logits [B*N][vocab]: the argmax of every
    row, then the greedy walk over it. Returns (target_argmax [B][N],
    accept_len [B], accepted_path [B][N], accepted_tokens [B][N])."""
    parents = np.asarray(parents)
    B, N = parents.shape
    arg = row_argmax(logits).reshape(B, N)
    alen, path, tok = _walk.greedy_walk_batch(parents, draft_tokens, arg)
    return arg, alen, path, tok
