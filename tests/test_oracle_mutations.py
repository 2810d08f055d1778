"""Planted mistakes in the oracle (on the CPU) must be caught by its pins.

Each case swaps one oracle function for a plausibly wrong version (a wrong
sign, a dropped term, an off-by-one, a transposed operand, the wrong tie rule)
and runs the pin that should catch it; the pin must then fail.
"""
import math

import numpy as np
import pytest

import oracle.attention as A
import oracle.compact as C
import oracle.fp8 as F8
import oracle.merge as M
import oracle.rope as R
import oracle.tree as T
import oracle.walk as W
from tests import test_oracle_attention as PA
from tests import test_oracle_fp8 as PF
from tests import test_oracle_tree as PT
from tests import test_oracle_walk_compact as PW
from tests.conftest import load_golden


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def _rope_wrong_sign(x, pos, theta):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * R.inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)


def _rope_adjacent_pairs(x, pos, theta):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * R.inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * c - x2 * s
    out[..., 1::2] = x2 * c + x1 * s
    return out


def test_rope_mutations_caught(monkeypatch):
    for bad in (_rope_wrong_sign, _rope_adjacent_pairs):
        monkeypatch.setattr(R, "rotate", bad)
        assert _fails(PA.test_rope_matches_complex_rotation)
        assert _fails(PA.test_chain_equals_causal_attention)


def test_attention_mutations_caught(monkeypatch):
    orig = A.verify_attention

    def no_scale(*a, **k):
        k["scale"] = 1.0
        return orig(*a, **k)
    monkeypatch.setattr(A, "verify_attention", no_scale)
    assert _fails(PA.test_chain_equals_causal_attention)
    monkeypatch.setattr(A, "verify_attention", orig)

    # query rotated at the node's index instead of its depth
    orig_root_path = A.root_path

    def q_at_index(parents, v):
        return list(range(v + 1)) if v < len(parents) else orig_root_path(parents, v)
    monkeypatch.setattr(A, "root_path", q_at_index)
    assert _fails(PA.test_each_node_is_its_own_root_path, [-1, 0, 0, 1, 2])
    monkeypatch.setattr(A, "root_path", orig_root_path)

    # wrong GQA mapping: head h reads KV head h % Hkv
    def mod_heads(q, k_new, v_new, k_cache, v_cache, *rest, **kw):
        g = q.shape[1] // rest[3]
        perm = np.arange(q.shape[1]).reshape(g, -1).T.reshape(-1)
        o, l = orig(q[:, perm], k_new, v_new, k_cache, v_cache, *rest, **kw)
        inv = np.argsort(perm)
        return o[:, inv], l[:, inv]
    monkeypatch.setattr(A, "verify_attention", mod_heads)
    assert _fails(PA.test_gqa_head_mapping_and_scale)


def test_tree_mutations_caught(monkeypatch):
    orig = T.ancestors
    monkeypatch.setattr(T, "ancestors", lambda p, i: orig(p, i)[1:] or [i])   # drops self
    assert _fails(PT.test_visibility_matrix_matches_page, load_golden)
    monkeypatch.setattr(T, "ancestors", orig)

    orig_links = T.links

    def links_descending(parents):
        n = len(parents)
        nt = np.full(n, -1, np.int32)
        ns = np.full(n, -1, np.int32)
        for p in range(n):
            kids = [j for j in range(n) if int(parents[j]) == p][::-1]
            if kids:
                nt[p] = kids[0]
            for a, b in zip(kids, kids[1:]):
                ns[a] = b
        return nt, ns
    monkeypatch.setattr(T, "links", links_descending)
    assert _fails(PT.test_links_examples, load_golden, "ddtree_retrieve.txt")
    monkeypatch.setattr(T, "links", orig_links)

    monkeypatch.setattr(T, "positions", lambda vc, depth: np.arange(len(depth)) + int(vc))
    assert _fails(PT.test_positions_examples, load_golden)


def test_walk_mutations_caught(monkeypatch):
    def last_match(parents, draft, argmax):
        parents = [int(x) for x in parents]
        n = len(parents)
        path, cur = [0], 0
        while True:
            m = [j for j in range(n) if parents[j] == cur and int(draft[j]) == int(argmax[cur])]
            if not m:
                break
            path.append(m[-1])
            cur = m[-1]
        ap = np.full(n, -1, np.int32)
        at = np.full(n, -1, np.int32)
        ap[: len(path)] = path
        at[: len(path)] = [int(argmax[u]) for u in path]
        return len(path), ap, at
    monkeypatch.setattr(W, "greedy_walk", last_match)
    assert _fails(PW.test_walk_with_duplicates_follows_the_definition, 4)

    def child_token_compared(parents, draft, argmax):   # compares argmax at the child
        parents = [int(x) for x in parents]
        n = len(parents)
        path, cur = [0], 0
        while True:
            m = [j for j in range(n) if parents[j] == cur and int(draft[j]) == int(argmax[j])]
            if not m:
                break
            path.append(m[0])
            cur = m[0]
        ap = np.full(n, -1, np.int32)
        at = np.full(n, -1, np.int32)
        ap[: len(path)] = path
        at[: len(path)] = [int(argmax[u]) for u in path]
        return len(path), ap, at
    monkeypatch.setattr(W, "greedy_walk", child_token_compared)
    assert _fails(PW.test_walk_examples, load_golden, "accept_0_2_5_6.txt")


def test_compact_and_merge_mutations_caught(monkeypatch):
    def in_place_descending(buffers, wl, path, alen):
        path = np.asarray(path)
        B, N = path.shape
        out = []
        for buf in buffers:
            new = np.array(buf, copy=True)
            for b in range(B):
                for t in reversed(range(int(alen[b]))):
                    new[wl[b * N + t]] = new[wl[b * N + int(path[b, t])]]
            out.append(new)
        return out
    monkeypatch.setattr(C, "compact_window_rows", in_place_descending)
    assert _fails(PW.test_compact_overlap_reads_before_writes)

    monkeypatch.setattr(M, "merge_states",
                        lambda outs, ls: (np.mean(np.asarray(outs, float), axis=0), np.max(ls, axis=0)))
    assert _fails(PA.test_merge_scalar_example, load_golden)
    assert math.isfinite(1.0)


def _argmax_last_of_ties(logits):
    x = np.asarray(logits)
    return (x.shape[1] - 1 - np.argmax(x[:, ::-1], axis=1)).astype(np.int32)


def _argmax_ignoring_nan(logits):
    x = np.asarray(logits, dtype=np.float64)
    x = np.where(np.isnan(x), -np.inf, x)
    return np.argmax(x, axis=1).astype(np.int32)


def _argmax_of_column(logits):  # a transposed operand: argmax down the columns
    x = np.asarray(logits)
    return np.resize(np.argmax(x, axis=0), x.shape[0]).astype(np.int32)


def test_argmax_mutations_caught(monkeypatch):
    import oracle.argmax as AM
    from tests import test_oracle_argmax as PM
    for bad in (_argmax_last_of_ties, _argmax_ignoring_nan, _argmax_of_column):
        monkeypatch.setattr(AM, "row_argmax", bad)
        caught = _fails(PM.test_matches_plain_scan_with_many_ties)
        for row, expect in ([[2.0, math.nan, 9.0, math.nan], 1], [[1.0, 7.0, 3.0, 7.0], 1]):
            caught = caught or _fails(PM.test_special_cases, row, expect)
        assert caught, bad.__name__


def test_window_attention_mutations_caught(monkeypatch):
    import oracle.attention as AT
    from tests import test_oracle_window as PW2
    real = AT.window_attention

    def shifted_mask(q, kc, vc, pt, plen, mask, pos, W, *a, **k):      # bit j read as key j + 1
        return real(q, kc, vc, pt, plen, [[(int(m) << 1) & ((1 << W) - 1) for m in row] for row in mask], pos, W,
                    *a, **k)

    def mask_ignored(q, kc, vc, pt, plen, mask, pos, W, *a, **k):      # every window key visible
        return real(q, kc, vc, pt, plen, [[(1 << W) - 1 for _ in row] for row in mask], pos, W, *a, **k)

    def position_by_row(q, kc, vc, pt, plen, mask, pos, W, *a, **k):   # the query at prefix + row index
        return real(q, kc, vc, pt, plen, mask, [[int(plen[b]) + r for r in range(len(row))]
                                                 for b, row in enumerate(pos)], W, *a, **k)

    for bad in (shifted_mask, mask_ignored, position_by_row):
        monkeypatch.setattr(AT, "window_attention", bad)
        caught = _fails(PW2.test_lane_rows_equal_tree_rows)
        caught = caught or _fails(PW2.test_equals_path_oracle_on_trees, [-1, 0, 0, 1, 2])
        assert caught, bad.__name__


def test_sampling_mutations_caught(monkeypatch):
    import oracle.sampling as SM
    from tests import test_oracle_sampling as PS
    real_scores, real_gumbel, real_draws = SM.sampled_scores, SM.gumbel_f32, SM.sampled_draws

    def draws_pos_without_plus_one(logits, vc, depth, temperature, seed):   # the node's own position
        depth = np.asarray(depth)
        return real_draws(logits, np.asarray(vc) - 1, depth, temperature, seed)

    def draws_keyed_by_row(logits, vc, depth, temperature, seed):
        depth = np.asarray(depth)
        B, N = depth.shape
        rows = np.tile(np.arange(N), (B, 1))
        return real_draws(logits, np.zeros(B, np.int64), rows, temperature, seed)

    def scores_ignore_temperature(x, temperature, seed, pos):
        return real_scores(x, 1.0 if temperature > 0 else temperature, seed, pos)

    def gumbel_log2(seed, pos, vocab):
        g = real_gumbel(seed, pos, vocab).astype(np.float64)
        # the same uniforms through -log2(-log2(u)) instead of -ln(-ln(u))
        u = np.exp(-np.exp(-g))
        return (-np.log2(-np.log2(u))).astype(np.float32)

    cases = [("sampled_draws", draws_pos_without_plus_one, PS.test_chain_accepts_plain_decoding_draws, ()),
             ("sampled_draws", draws_keyed_by_row, PS.test_keyed_by_position_not_row, ()),
             ("sampled_scores", scores_ignore_temperature, PS.test_draws_follow_softmax, (0.7,)),
             ("gumbel_f32", gumbel_log2, PS.test_draws_follow_softmax, (1.0,))]
    for name, bad, pin, args in cases:
        monkeypatch.setattr(SM, name, bad)
        assert _fails(pin, *args), bad.__name__
        monkeypatch.undo()


def _decode_bias8(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e, m = (c >> 3) & 0xF, c & 0x7
    v = np.where(e == 0, np.ldexp(m / 8.0, -7), np.ldexp(1.0 + m / 8.0, e - 8))
    v = np.where(c & 0x80, -v, v)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def _decode_ieee_specials(codes):  # exponent 15 reserved for inf/NaN, as in IEEE formats
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    v = _ORIG_DECODE(codes)
    return np.where(((c >> 3) & 0xF) == 0xF, np.nan, v)


def _decode_subnormal_no_scale(codes):  # subnormals read as 2^-7 * m / 8 (the normal formula with e = 0)
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    v = _ORIG_DECODE(codes)
    e, m = (c >> 3) & 0xF, c & 0x7
    sub = np.where(c & 0x80, -1.0, 1.0) * np.ldexp(1.0 + m / 8.0, -7)
    return np.where((e == 0) & (m != 0), sub, v)


_ORIG_DECODE = F8.decode_e4m3
_ORIG_ENCODE = F8.encode_e4m3


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    out = _ORIG_ENCODE(x)
    grid = _ORIG_DECODE(np.arange(0x7F, dtype=np.uint8))
    a = np.abs(x)
    hi = np.clip(np.searchsorted(grid, a), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    tie = (a - grid[lo]) == (grid[hi] - a)
    return np.where(tie & (a < 448), (hi | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8), out)


def _encode_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    grid = _ORIG_DECODE(np.arange(0x7F, dtype=np.uint8))
    a = np.minimum(np.abs(x), 448.0)
    code = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, 0x7E)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def _encode_nan_on_overflow(x):
    x = np.asarray(x, dtype=np.float64)
    return np.where(np.abs(x) >= 464, np.uint8(0x7F), _ORIG_ENCODE(x)).astype(np.uint8)


def test_fp8_mutations_caught(monkeypatch):
    for bad in (_decode_bias8, _decode_ieee_specials, _decode_subnormal_no_scale):
        monkeypatch.setattr(F8, "decode_e4m3", bad)
        assert _fails(PF.test_decode_fixed_points) or _fails(PF.test_decode_matches_torch_on_every_code)
        monkeypatch.setattr(F8, "decode_e4m3", _ORIG_DECODE)
    for bad in (_encode_ties_away, _encode_truncate, _encode_nan_on_overflow):
        monkeypatch.setattr(F8, "encode_e4m3", bad)
        assert _fails(PF.test_encode_matches_torch_below_saturation) or _fails(PF.test_encode_ties_to_even_and_saturates)
        monkeypatch.setattr(F8, "encode_e4m3", _ORIG_ENCODE)


def test_fp8_query_split_mutations_caught(monkeypatch):
    """The E4M3 query cast applied to the window keys as well, or to no key,
    fails the pin that separates the two parts."""
    import oracle.attention as AT
    from tests import test_oracle_window as PW2
    real_prefix = AT.prefix_query

    def window_cast(qv, q_fp8):                # the window keys also see the cast query
        return F8.decode_e4m3(F8.encode_e4m3(qv)) if q_fp8 else qv

    def no_cast(qv, q_fp8):                    # the prefix keys see the unquantized query
        return qv

    for name, bad in (("window_query", window_cast), ("prefix_query", no_cast)):
        monkeypatch.setattr(AT, name, bad)
        assert _fails(PW2.test_fp8_query_scores_the_prefix_only), name
        monkeypatch.undo()
    assert AT.prefix_query is real_prefix
