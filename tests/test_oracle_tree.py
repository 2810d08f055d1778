"""Pins for oracle.tree: values the pages print, brute force and invariants."""
import itertools

import numpy as np
import pytest

from oracle import tree as T


def _all_trees(n):
    """Every parent array with parents[0] = -1 and 0 <= parents[i] < i."""
    for rest in itertools.product(*[range(i) for i in range(1, n)]):
        yield [-1, *rest]


def _closure_by_matrix_powers(parents):
    """Reachability child -> ancestor by repeated boolean matrix products
    (an independent way to get the ancestor sets: no parent walk)."""
    n = len(parents)
    A = np.zeros((n, n), dtype=bool)
    for i, p in enumerate(parents):
        if p >= 0:
            A[i, p] = True
    R = np.eye(n, dtype=bool)
    step = np.eye(n, dtype=bool)
    for _ in range(n):
        step = (step.astype(int) @ A.astype(int)) > 0
        R |= step
    return R


def test_visibility_matrix_matches_page(golden):
    g = golden("visibility_root_abcd.txt")
    vis = T.visibility_matrix(g["parents"])
    want = np.array([[int(c) for c in row] for row in g["tree_visibility"]])
    assert (vis == want).all()


def test_chain_is_lower_triangular(golden):
    g = golden("visibility_root_abcd.txt")
    parents = [-1, 0, 1, 2, 3]                      # the chain parent[i] = i - 1
    want = np.array([[int(c) for c in row] for row in g["causal_visibility"]])
    assert (T.visibility_matrix(parents) == want).all()
    for n in (1, 2, 17, 64):
        assert (T.visibility_matrix(list(range(-1, n - 1))) == np.tril(np.ones((n, n), int))).all()


def test_toy_closure_row(golden):
    g = golden("toy_closure.txt")
    vis = T.visibility_matrix(g["parents"])
    assert vis[2].tolist() == g["mask_row_2"]


def test_bit63_and_full_width():
    chain = list(range(-1, 63))
    m = T.ancestor_mask(chain)
    assert int(m[63]) == (1 << 64) - 1
    star = [-1] + [0] * 63
    m = T.ancestor_mask(star)
    assert int(m[63]) == (1 << 63) | 1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_mask_brute_force_all_trees(n):
    for parents in _all_trees(n):
        R = _closure_by_matrix_powers(parents)
        m = T.ancestor_mask(parents)
        depth = [len(T.ancestors(parents, i)) - 1 for i in range(n)]
        for i in range(n):
            bits = [(int(m[i]) >> j) & 1 for j in range(n)]
            assert bits == R[i].astype(int).tolist()
            assert bin(int(m[i])).count("1") == depth[i] + 1
            if i:
                assert int(m[i]) == int(m[parents[i]]) | (1 << i)
            assert int(m[i]) >> n == 0


def test_positions_examples(golden):
    g = golden("positions_depth_prefix7.txt")
    assert T.positions(g["prefix_len"][0], g["depth"]).tolist() == g["positions"]
    g = golden("links_build_eagle_tree.txt")
    depth = [len(T.ancestors(g["parents"], i)) - 1 for i in range(len(g["parents"]))]
    assert T.positions(g["prefix_len"][0], depth).tolist() == g["positions"]


@pytest.mark.parametrize("name", ["links_build_eagle_tree.txt", "ddtree_retrieve.txt"])
def test_links_examples(golden, name):
    g = golden(name)
    nt, ns = T.links(g["parents"])
    assert nt.tolist() == g["next_token"]
    assert ns.tolist() == g["next_sibling"]


@pytest.mark.parametrize("n", [1, 3, 5, 6])
def test_links_traversal_covers_each_node_once(n):
    for parents in _all_trees(n):
        nt, ns = T.links(parents)
        seen = []

        def visit(u):
            seen.append(u)
            c = nt[u]
            while c != -1:
                assert parents[c] == u
                visit(c)
                c = ns[c]
        visit(0)
        assert sorted(seen) == list(range(n))
        # depth-first order with children in ascending index is 0..n-1 exactly when
        # the tree is numbered depth first
        for i in range(n):
            kids = [j for j in range(n) if parents[j] == i]
            assert kids == sorted(kids)


def test_validation():
    assert T.tree_error([-1, 0, 0, 1, 2], [0, 1, 1, 2, 2]) is None
    assert T.tree_error([0, 0], None) == "bad_parent"
    assert T.tree_error([-1, 1], None) == "bad_parent"          # self parent
    assert T.tree_error([-1, 2, 0], None) == "bad_parent"       # parent after child
    assert T.tree_error([-1, -1], None) == "bad_parent"         # second root (a forest)
    assert T.tree_error([-1, 0, 1], [0, 1, 1]) == "bad_depth"
    assert T.tree_error([-1, 0], [1, 2]) == "bad_depth"
    assert T.tree_error([], None) == "unsupported_size"
    assert T.tree_error([-1] + [0] * 64, None) == "unsupported_size"
    with pytest.raises(ValueError):
        T.build_tree_mask([-1, 0, 1], [0, 1, 3], 0)


def test_toy_selection_closure(golden):
    """The page's ranking (-score, depth, id) keeps an ancestor-closed set."""
    g = golden("toy_closure.txt")
    parents, scores = g["parents"], g["scores"]
    depth = [len(T.ancestors(parents, i)) - 1 for i in range(len(parents))]
    ranked = sorted(range(1, len(parents)), key=lambda i: (-scores[i], depth[i], i))
    sel = {0, *ranked[:2]}
    assert sorted(sel) == g["selected"]
    assert all(parents[i] in sel for i in sel if i)
    bad = set(g["not_closed"])
    assert any(parents[i] not in bad for i in bad if i)
