"""Pins for oracle.walk and oracle.compact."""
import itertools

import numpy as np
import pytest

from oracle import compact as C
from oracle import tree as T
from oracle import walk as W


def _all_trees(n):
    for rest in itertools.product(*[range(i) for i in range(1, n)]):
        yield [-1, *rest]


def _root_paths(parents):
    n = len(parents)
    return [T.root_path(parents, v) for v in range(n)]


@pytest.mark.parametrize("name", ["accept_0_2_5_6.txt", "chain_walk.txt"])
def test_walk_examples(golden, name):
    g = golden(name)
    alen, path, tok = W.greedy_walk(g["parents"], g["draft"], g["target_argmax"])
    assert alen == g["accept_len"][0]
    assert path[: len(g["accepted_path"])].tolist() == g["accepted_path"]
    assert tok[: len(g["accepted_tokens"])].tolist() == g["accepted_tokens"]
    assert (path[alen:] == -1).all() and (tok[alen:] == -1).all()


def test_chain_accepts_one_plus_leading_matches():
    rng = np.random.default_rng(11)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        parents = list(range(-1, n - 1))
        argmax = rng.integers(0, 3, n)
        draft = rng.integers(0, 3, n)
        lead = 0
        for i in range(1, n):
            if draft[i] == argmax[i - 1]:
                lead += 1
            else:
                break
        alen, path, tok = W.greedy_walk(parents, draft, argmax)
        assert alen == 1 + lead
        assert path[:alen].tolist() == list(range(alen))


@pytest.mark.parametrize("n", [2, 3, 4, 5, 6])
def test_walk_brute_force_distinct_sibling_tokens(n):
    """With distinct tokens among siblings, the result is the unique longest
    root path whose every edge matches (child's draft == parent's argmax)."""
    rng = np.random.default_rng(12 + n)
    for parents in _all_trees(n):
        argmax = rng.integers(0, 4, n)
        draft = np.zeros(n, int)
        for p in range(n):
            kids = [j for j in range(n) if parents[j] == p]
            toks = rng.permutation(6)[: len(kids)]      # distinct among siblings
            for j, t in zip(kids, toks):
                draft[j] = t
        full = [pth for pth in _root_paths(parents)
                if all(draft[pth[t]] == argmax[pth[t - 1]] for t in range(1, len(pth)))]
        best = max(len(p) for p in full)
        longest = [p for p in full if len(p) == best]
        assert len(longest) == 1
        alen, path, tok = W.greedy_walk(parents, draft, argmax)
        assert path[:alen].tolist() == longest[0]
        assert tok[:alen].tolist() == [int(argmax[u]) for u in longest[0]]


@pytest.mark.parametrize("n", [3, 4, 5, 6])
def test_walk_with_duplicates_follows_the_definition(n):
    """With repeated sibling tokens: the path matches on every edge, nothing
    extends it, and no lower-index sibling of an accepted node also matched."""
    rng = np.random.default_rng(30 + n)
    for parents in _all_trees(n):
        argmax = rng.integers(0, 2, n)
        draft = rng.integers(0, 2, n)
        alen, path, _ = W.greedy_walk(parents, draft, argmax)
        p = path[:alen].tolist()
        depth = [len(T.ancestors(parents, i)) - 1 for i in range(n)]
        assert p[0] == 0
        for t in range(1, alen):
            assert parents[p[t]] == p[t - 1] and draft[p[t]] == argmax[p[t - 1]]
            assert depth[p[t]] == t
            assert not any(parents[j] == p[t - 1] and draft[j] == argmax[p[t - 1]]
                           for j in range(p[t]))
        assert not any(parents[j] == p[-1] and draft[j] == argmax[p[-1]] for j in range(n))


def test_compact_example_slots_0_2_5_6(golden):
    g = golden("accept_0_2_5_6.txt")
    N = 8
    rng = np.random.default_rng(13)
    buf = rng.integers(0, 256, (N + 4, 12), dtype=np.uint8)
    wl = np.arange(N)                        # the 8-slot block at slots 0..7
    path = np.array([g["accepted_path"]])
    new, = C.compact_window_rows([buf], wl, path, [g["accept_len"][0]])
    for t, s in enumerate(g["moved_slots"]):
        assert (new[t] == buf[s]).all()
    assert (new[4:] == buf[4:]).all()        # rejected slots and the rest: unchanged


def test_compact_overlap_reads_before_writes():
    rng = np.random.default_rng(14)
    buf = rng.integers(0, 256, (6, 8), dtype=np.uint8)
    wl = np.array([2, 3, 4, 5])              # window of 4 starting at slot 2
    new, = C.compact_window_rows([buf], wl, np.array([[0, 2, 3, -1]]), [3])
    assert (new[2] == buf[2]).all() and (new[3] == buf[4]).all() and (new[4] == buf[5]).all()
    assert (new[[0, 1, 5]] == buf[[0, 1, 5]]).all()
    # a sequential in-place copy in ascending t gives the same answer for
    # strictly increasing paths; a copy that writes t = 2 first does not
    bad = buf.copy()
    bad[4] = bad[5]
    bad[3] = bad[4]
    assert not (bad[3] == new[3]).all()


def test_compact_identity_cases():
    rng = np.random.default_rng(15)
    buf = rng.integers(0, 256, (10, 16), dtype=np.uint8)
    wl = np.arange(2, 10)
    chain = np.arange(8)[None]
    assert (C.compact_window_rows([buf], wl, chain, [8])[0] == buf).all()   # fresh chain
    one = np.array([[0] + [-1] * 7])
    assert (C.compact_window_rows([buf], wl, one, [1])[0] == buf).all()     # accept_len 1
    h = rng.integers(0, 256, (8, 6), dtype=np.uint8)
    assert (C.compact_hidden_rows(h, chain, [8]) == h).all()


def test_hidden_rows_gather():
    rng = np.random.default_rng(16)
    B, N = 2, 5
    h = rng.integers(0, 256, (B * N, 4), dtype=np.uint8)
    path = np.array([[0, 2, 4, -1, -1], [0, 1, -1, -1, -1]])
    new = C.compact_hidden_rows(h, path, [3, 2])
    assert (new[0] == h[0]).all() and (new[1] == h[2]).all() and (new[2] == h[4]).all()
    assert (new[3:5] == h[3:5]).all() and (new[5:] == h[5:]).all()


def test_position_shifts_cancel_for_any_depth():
    rng = np.random.default_rng(17)
    for _ in range(50):
        B, N = 3, int(rng.integers(1, 65))
        vc = rng.integers(0, 1 << 20, B)
        depth = rng.integers(0, N, (B, N))
        loaded = C.load_step_positions(vc, depth)
        assert (loaded - vc[:, None] == depth).all()
        back = C.compact_positions(vc, N)
        assert (back == vc[:, None] + np.arange(N)).all()
    # the fresh spec is the chain: depth = i gives the same positions both ways
    vc = np.array([7, 0])
    chain_depth = np.tile(np.arange(5), (2, 1))
    assert (C.load_step_positions(vc, chain_depth) == C.compact_positions(vc, 5)).all()
