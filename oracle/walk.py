"""Oracle: greedy tree verification, the naive walk straight from parents.

Test infrastructure only (see the package docstring).

Sources:
* [MI] "Walking the accepted path": start at the root; descend to the first
  child; scan its siblings for one whose draft token equals the target's
  argmax at the parent; accept it and repeat; stop when no sibling matches.
  The example there: nodes 0, 2, 5, 6 accept, accept_lens = 4,
  accept_index = [0, 2, 5, 6, -1, -1].
* [AK] section two: accept_lens = correct drafts + 1; the accepted outputs
  are the target's argmax at each accepted node (the last one is the bonus).
* [TS] "The tree is a parameter of the chain path": the accepted path is
  packed at the front.

Readings taken: children are scanned in ascending node index and the first
match wins (several siblings can carry the same token); the packed path and
tokens are N wide, padded with -1; node ids are local to the request.
"""
from __future__ import annotations

import numpy as np


def greedy_walk(parents, draft_tokens, target_argmax):
    """One request. Returns (accept_len, accepted_path int32[N], accepted_tokens int32[N])."""
    parents = [int(x) for x in parents]
    n = len(parents)
    path = [0]
    cur = 0
    while True:
        nxt = -1
        for j in range(n):                       # children of cur, ascending index
            if parents[j] == cur and int(draft_tokens[j]) == int(target_argmax[cur]):
                nxt = j
                break
        if nxt < 0:
            break
        path.append(nxt)
        cur = nxt
    acc_path = np.full(n, -1, dtype=np.int32)
    acc_tok = np.full(n, -1, dtype=np.int32)
    acc_path[: len(path)] = path
    acc_tok[: len(path)] = [int(target_argmax[u]) for u in path]
    return len(path), acc_path, acc_tok


def greedy_walk_batch(parents, draft_tokens, target_argmax):
    parents = np.asarray(parents)
    B, N = parents.shape
    alen = np.zeros(B, np.int32)
    apath = np.zeros((B, N), np.int32)
    atok = np.zeros((B, N), np.int32)
    for b in range(B):
        alen[b], apath[b], atok[b] = greedy_walk(parents[b], draft_tokens[b], target_argmax[b])
    return alen, apath, atok
