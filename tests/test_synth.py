"""The seeded input generator: deterministic, and its trees are valid verify trees."""
import numpy as np
import pytest

from draft_tree_speculative_gb300 import synth as S
from oracle import tree as T


@pytest.mark.parametrize("name", list(S.WORKLOADS))
def test_trees_are_valid_and_depth_first(name):
    w = S.WORKLOADS[name]
    parents, depth = S.make_trees(w, S.streams(w.index)["tree"])
    assert parents.shape == (w.B, w.N)
    for b in range(w.B):
        assert T.tree_error(parents[b], depth[b]) is None
        if w.tree == "fixed_root_abcd":     # the page's [root, A, B, C, D] is level order
            continue
        # depth-first numbering: every subtree occupies a contiguous index range
        n = w.N
        size = np.ones(n, int)
        for i in range(n - 1, 0, -1):
            size[parents[b, i]] += size[i]
        for i in range(n):
            sub = [j for j in range(n) if i in T.ancestors(parents[b], j)]
            assert sub == list(range(i, i + size[i]))
    if w.tree == "eagle2":
        assert depth.max() <= w.steps


def test_generator_is_deterministic():
    w = S.WORKLOADS["tiny_p128_n5"]
    a = S.make_inputs(w)
    b = S.make_inputs(w)
    assert (a.q == b.q).all() and (a.k_cache == b.k_cache).all() and (a.draft == b.draft).all()
    assert a.layout.page_table.tolist() == [[1, 2, 3]]


def test_layout_pages_are_disjoint_and_skip_page_zero():
    w = S.WORKLOADS["highconc_b128_n16"]
    s = S.streams(w.index)
    plen = S.make_prefix_lens(w, s["prefix"])
    assert plen.min() >= 512 and plen.max() <= 4096
    lay = S.make_layout(w, plen, s["pages"])
    used = []
    for b in range(w.B):
        need = (int(plen[b]) + w.N + 63) // 64
        used += lay.page_table[b, :need].tolist()
        assert (lay.page_table[b, need:] == 0).all()
    assert 0 not in used and len(set(used)) == len(used)
    assert len(set(lay.write_locations.tolist())) == w.B * w.N


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 65504.0], np.float32)
    got = S.bf16_bits_to_f64(S.f32_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 65536.0]


def test_e4m3_draws_are_finite_and_normal_shaped():
    """normal_e4m3: no NaN code, both signs, and the decoded draws keep the
    N(0,1) shape (each value is the draw with its mantissa cut to three bits,
    so within 12.5% below it in magnitude)."""
    from oracle import fp8 as F8
    rng = np.random.default_rng(0)
    codes = S.normal_e4m3(rng, (200000,))
    assert ((codes & 0x7F) != 0x7F).all()
    x = F8.decode_e4m3(codes)
    assert abs(x.mean()) < 0.01 and 0.85 < x.std() < 1.0
    assert (x > 0).mean() > 0.49 and (x < 0).mean() > 0.49
    ref = np.random.default_rng(0).standard_normal(200000, dtype=np.float32).astype(np.float64)
    big = np.abs(ref) >= 2.0 ** -6
    assert (np.abs(x[big]) <= np.abs(ref[big])).all() and (np.abs(x[big]) > 0.875 * np.abs(ref[big])).all()
    assert (x[~big] == 0).all()
