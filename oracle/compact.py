"""Oracle: compaction of the accepted path (KV rows, hidden rows, positions).

Test infrastructure only (see the package docstring).

Sources:
* [TS] "The tree is a parameter of the chain path": the path's target KV of
  every layer moves to the window's leading slots by a word copy that does
  not care about dtype; the hidden rows move to the front of the window and
  the positions go back from vc + depth to vc + i.
* [TS] "Position follows depth, slot follows node index": node i's KV slot is
  write_locations[b * N + i]; the two position shifts cancel for any depth.
* [MI] "Discarding the rejected branches' KV": destinations are the first
  accept_len window slots, sources are the accepted nodes' slots; rejected
  slots are left as they are.

Reading taken: the move is a gather of a snapshot followed by a scatter, so an
accepted row that is also a destination (path [0, 2, 3]: slot 2 is read for
t = 1 and written for t = 2) is read before it is overwritten.
"""
from __future__ import annotations

import numpy as np


def compact_window_rows(buffers, write_locations, accepted_path, accept_len):
    """buffers: list of uint8 arrays [num_slots][row_bytes] (any row size).
    Returns new arrays; the inputs are not modified."""
    accepted_path = np.asarray(accepted_path)
    B, N = accepted_path.shape
    wl = np.asarray(write_locations, dtype=np.int64)
    out = []
    for buf in buffers:
        snap = np.array(buf, copy=True)
        new = np.array(buf, copy=True)
        for b in range(B):
            for t in range(int(accept_len[b])):
                dst = wl[b * N + t]
                src = wl[b * N + int(accepted_path[b, t])]
                new[dst] = snap[src]
        out.append(new)
    return out


def compact_hidden_rows(hidden, accepted_path, accept_len):
    """hidden: [B*N][row_bytes]; row b*N + t <- snapshot row b*N + path[t]."""
    accepted_path = np.asarray(accepted_path)
    B, N = accepted_path.shape
    snap = np.array(hidden, copy=True)
    new = np.array(hidden, copy=True)
    for b in range(B):
        for t in range(int(accept_len[b])):
            new[b * N + t] = snap[b * N + int(accepted_path[b, t])]
    return new


def load_step_positions(vc, depth):
    """Before the forward: window positions vc + i -> vc + depth[i]."""
    vc = np.asarray(vc, dtype=np.int64)
    return np.asarray(depth, dtype=np.int64) + vc[:, None]


def compact_positions(vc, N: int):
    """After the forward: every window row i goes back to vc + i."""
    vc = np.asarray(vc, dtype=np.int64)
    return vc[:, None] + np.arange(N, dtype=np.int64)[None, :]
