"""Oracle: tree validation, 64-bit ancestor mask, positions and child links.

Test infrastructure only (see the package docstring).

Sources:
* [TS] "Draft-tree speculation", sections "The tree is a parameter of the chain
  path" (a chain is parent[i] = i - 1), "Position follows depth, slot follows
  node index" (position = vc + depth[i]) and "One tree attention" (one 64-bit
  ancestor mask per row, N <= 64).
* [AK] section one (visibility: committed prefix, the node itself and its
  ancestors; nothing else) and section two (siblings share a position).
* [MI] "Flattening, and the two link arrays" (first-child / next-sibling
  encoding).
"""
from __future__ import annotations

from typing import Optional

import numpy as np

MAX_NODES = 64


def tree_error(parents, depth=None) -> Optional[str]:
    """None if (parents, depth) is a valid verify tree, else the reason.

    Reading taken where the pages are silent: node 0 is the root (parent -1),
    every other node's parent has a smaller index (depth-first numbering puts
    parents first), and depth, when given, must equal the parent's depth + 1.
    """
    parents = [int(x) for x in parents]
    n = len(parents)
    if n < 1 or n > MAX_NODES:
        return "unsupported_size"
    if parents[0] != -1:
        return "bad_parent"
    for i in range(1, n):
        if not (0 <= parents[i] < i):
            return "bad_parent"
    if depth is not None:
        depth = [int(x) for x in depth]
        if depth[0] != 0:
            return "bad_depth"
        for i in range(1, n):
            if depth[i] != depth[parents[i]] + 1:
                return "bad_depth"
    return None


def ancestors(parents, i: int) -> list:
    """Node i and every ancestor up to the root, found by walking parent links
    (this never reads depth)."""
    out = []
    j = int(i)
    while j != -1:
        out.append(j)
        j = int(parents[j])
    return out


def root_path(parents, v: int) -> list:
    """u_0 = root, ..., u_D = v."""
    return list(reversed(ancestors(parents, v)))


def ancestor_mask(parents) -> np.ndarray:
    """mask[i] has bit j set iff j == i or j is an ancestor of i ([AK] §1)."""
    n = len(parents)
    m = np.zeros(n, dtype=np.uint64)
    for i in range(n):
        bits = 0
        for j in ancestors(parents, i):
            bits |= 1 << j
        m[i] = np.uint64(bits)
    return m


def visibility_matrix(parents) -> np.ndarray:
    """The window part of [AK] §1's visibility matrix: vis[i, j] = bit j of mask[i]."""
    m = ancestor_mask(parents)
    n = len(parents)
    return np.array([[(int(m[i]) >> j) & 1 for j in range(n)] for i in range(n)], dtype=np.int32)


def positions(vc: int, depth) -> np.ndarray:
    """RoPE position of node i: vc + depth[i] ([TS] "Position follows depth")."""
    return np.asarray(depth, dtype=np.int64) + int(vc)


def links(parents):
    """First-child / next-sibling links ([MI] "Flattening, and the two link
    arrays"). Children of a node are ordered by ascending node index, which under
    depth-first best-child-first numbering is descending draft score."""
    n = len(parents)
    next_token = np.full(n, -1, dtype=np.int32)
    next_sibling = np.full(n, -1, dtype=np.int32)
    for p in range(n):
        kids = [j for j in range(n) if int(parents[j]) == p]
        if kids:
            next_token[p] = kids[0]
        for a, b in zip(kids, kids[1:]):
            next_sibling[a] = b
    return next_token, next_sibling


def build_tree_mask(parents, depth, vc: int):
    """Everything the mask-building step returns for one request:
    (mask u64[N], positions int64[N], next_token int32[N], next_sibling int32[N]).
    Raises ValueError with the reason for an invalid tree."""
    err = tree_error(parents, depth)
    if err is not None:
        raise ValueError(err)
    nt, ns = links(parents)
    return ancestor_mask(parents), positions(vc, depth), nt, ns
