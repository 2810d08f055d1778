"""Pins for oracle.attention.window_attention (R query rows over the prefix
plus a masked window of W cache keys: verify with R = W = N, draft lanes with
R = K rows over the (S - 1) * K-key lane window).

It is checked against the path-driven verify oracle (a different statement of
the same attention: keys gathered by walking parents, window keys rotated
from k_new) on trees and on a lane tree, against the independent causal
attention for a chain, and against closed forms."""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import rope as Rr
from oracle import tree as T
from tests.test_oracle_attention import THETA, _case, _prefix_seq, causal_attention, rope_complex


def _depth(parents):
    return [len(T.root_path(parents, v)) - 1 for v in range(len(parents))]


def _write_window(kc, table, P, page, kn_rows, depth, b=0):
    """The cache after the verify prologue: node i's K, rotated at P + depth[i],
    in the slot of logical position P + i (exact rotation: these pins use fp64)."""
    kc = kc.copy()
    sl = A.prefix_slots(table[b], P + len(depth), page)
    for i, dep in enumerate(depth):
        kc[sl[P + i]] = Rr.rotate(kn_rows[i], P + dep, THETA)
    return kc


def _write_values(vc, table, P, page, vn_rows, b=0):
    vc = vc.copy()
    sl = A.prefix_slots(table[b], P + len(vn_rows), page)
    for i in range(len(vn_rows)):
        vc[sl[P + i]] = vn_rows[i]
    return vc


@pytest.mark.parametrize("parents", [[-1, 0, 0, 1, 2], [-1, 0, 1, 2, 3, 4], [-1, 0, 0, 0, 1, 1, 4]])
def test_equals_path_oracle_on_trees(parents):
    rng = np.random.default_rng(50 + len(parents))
    N, Hq, Hkv, d, P, page = len(parents), 4, 2, 16, 9, 4
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, P, parents, page)
    depth = _depth(parents)
    kc2 = _write_window(kc, table, P, page, kn, depth)
    vc2 = _write_values(vc, table, P, page, vn)
    mask = [[int(T.ancestor_mask(parents)[i]) for i in range(N)]]
    pos = [[P + int(x) for x in depth]]
    out, lse = A.window_attention(q, kc2, vc2, table, plen, mask, pos, N, Hkv, THETA, page_size=page, rope_out=None)
    ref_o, ref_l = A.verify_attention(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page, rope_out=None)
    assert np.allclose(out, ref_o, atol=1e-12) and np.allclose(lse, ref_l, atol=1e-12)


def test_lane_rows_equal_tree_rows():
    """Draft lanes: K lanes over S - 1 steps form a tree (each lane of step s
    has a parent lane at step s - 1); lane row r of the last step, attending
    with its lane mask over the (S - 1) * K window, equals verify row
    (S - 2) * K + r of that tree. R = K != W here."""
    rng = np.random.default_rng(61)
    K, S = 3, 4
    W = (S - 1) * K
    parents = [-1] * W
    for s in range(1, S - 1):
        for r in range(K):
            parents[s * K + r] = (s - 1) * K + int(rng.integers(0, K))
    # step 1's K lanes have no window ancestor: the tree gets a virtual root
    # (node 0) that no lane row sees, and window key j is tree node j + 1
    Hq, Hkv, d, P, page = 4, 2, 16, 7, 4
    tree = [-1] + [p + 1 if p >= 0 else 0 for p in parents]
    N = len(tree)
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, P, tree, page)
    depth = _depth(tree)
    # window slot j holds tree node j + 1, rotated at P + depth - 1 (its lane step)
    kc2 = kc.copy()
    vc2 = vc.copy()
    sl = A.prefix_slots(table[0], P + W + 1, page)
    for j in range(W):
        kc2[sl[P + j]] = Rr.rotate(kn[j + 1], P + depth[j + 1] - 1, THETA)
        vc2[sl[P + j]] = vn[j + 1]
    anc = T.ancestor_mask(tree)
    lane_rows = [(S - 2) * K + r for r in range(K)]
    mask = [[int(anc[j + 1]) >> 1 for j in lane_rows]]            # drop the virtual root's bit
    pos = [[P + int(depth[j + 1]) - 1 for j in lane_rows]]
    qr = q[[j + 1 for j in lane_rows]]
    out, lse = A.window_attention(qr, kc2, vc2, table, plen, mask, pos, W, Hkv, THETA, page_size=page,
                                  rope_out=None)
    # the reference: each lane row's keys as an explicit sequence through the
    # independent causal attention (prefix, then the lane's ancestors in step
    # order, the lane's own token last, each at position P + step - 1)
    kp, vp = _prefix_seq(kc, vc, table, 0, P, page)
    for r, j in enumerate(lane_rows):
        path = T.root_path(tree, j + 1)[1:]                       # window nodes, step order
        k_seq = np.concatenate([kp, kn[path]])
        v_seq = np.concatenate([vp, vn[path]])
        q_seq = np.concatenate([np.zeros((P, Hq, d)), np.zeros((len(path) - 1, Hq, d)), q[[j + 1]]])
        ref_o, ref_l = causal_attention(q_seq, k_seq, v_seq, P, THETA, Hkv)
        assert np.allclose(out[r], ref_o[-1], atol=1e-10)
        assert np.allclose(lse[r], ref_l[-1], atol=1e-10)


def test_chain_equals_causal_attention():
    rng = np.random.default_rng(62)
    N, Hq, Hkv, d, P, page = 6, 4, 2, 16, 5, 4
    parents = list(range(-1, N - 1))
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, P, parents, page)
    depth = list(range(N))
    kc2 = _write_window(kc, table, P, page, kn, depth)
    vc2 = _write_values(vc, table, P, page, vn)
    mask = [[(1 << (i + 1)) - 1 for i in range(N)]]
    pos = [[P + i for i in range(N)]]
    out, lse = A.window_attention(q, kc2, vc2, table, plen, mask, pos, N, Hkv, THETA, page_size=page, rope_out=None)
    kp, vp = _prefix_seq(kc, vc, table, 0, P, page)
    q_seq = np.concatenate([np.zeros((P, Hq, d)), q])
    ref_o, ref_l = causal_attention(q_seq, np.concatenate([kp, kn]), np.concatenate([vp, vn]), P, THETA, Hkv)
    assert np.allclose(out, ref_o, atol=1e-10) and np.allclose(lse, ref_l, atol=1e-10)


def test_single_visible_key_and_nothing_visible():
    rng = np.random.default_rng(63)
    Hq, Hkv, d, page, W = 2, 1, 8, 4, 5
    table = np.array([[3, 1, 2]])
    kc = rng.standard_normal((16, Hkv, d))
    vc = rng.standard_normal((16, Hkv, d))
    q = rng.standard_normal((2, Hq, d))
    j = 3
    out, lse = A.window_attention(q, kc, vc, table, [0], [[1 << j, 0]], [[9, 9]], W, Hkv, THETA, page_size=page,
                                  rope_out=None)
    slot = A.prefix_slots(table[0], W, page)[j]
    qr = Rr.rotate(q[0], 9, THETA)
    for h in range(Hq):
        assert np.allclose(out[0, h], vc[slot, 0])                 # softmax over one key is 1
        assert math.isclose(lse[0, h], (qr[h] @ kc[slot, 0]) / math.sqrt(d) / math.log(2.0), rel_tol=1e-12)
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()       # no key at all (P = 0, empty mask)


def test_window_order_is_irrelevant():
    """Permuting the window slots together with the mask bits changes nothing:
    the rows see a set of keys."""
    rng = np.random.default_rng(64)
    Hq, Hkv, d, page, W, P, R = 4, 2, 16, 4, 7, 6, 3
    need = (P + W + page - 1) // page
    table = rng.permutation(np.arange(1, need + 1))[None]
    slots = (need + 1) * page
    kc = rng.standard_normal((slots, Hkv, d))
    vc = rng.standard_normal((slots, Hkv, d))
    q = rng.standard_normal((R, Hq, d))
    masks = [int(x) for x in rng.integers(0, 1 << W, R)]
    pos = [[P + 3] * R]
    out, lse = A.window_attention(q, kc, vc, table, [P], [masks], pos, W, Hkv, THETA, page_size=page)
    perm = rng.permutation(W)
    sl = A.prefix_slots(table[0], P + W, page)
    kc2, vc2 = kc.copy(), vc.copy()
    for j in range(W):
        kc2[sl[P + perm[j]]] = kc[sl[P + j]]
        vc2[sl[P + perm[j]]] = vc[sl[P + j]]
    masks2 = [sum(1 << int(perm[j]) for j in range(W) if (m >> j) & 1) for m in masks]
    out2, lse2 = A.window_attention(q, kc2, vc2, table, [P], [masks2], pos, W, Hkv, THETA, page_size=page)
    assert np.allclose(out, out2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)


def test_fp8_cache_reads_the_values_its_bytes_encode():
    """kv_fp8: a cache of E4M3 bytes attends exactly like a bf16 cache holding
    the same values (every E4M3 value is a bf16 value, so the bf16 cache is
    exact). The bytes cover subnormals, both signs and the largest finite code;
    a wrong decode, or K and V swapped, moves the result."""
    from oracle import fp8 as F8
    rng = np.random.default_rng(91)
    B, R, W, Hq, Hkv, d, page = 2, 3, 5, 4, 2, 16, 4
    P = [7, 0]
    slots = 64
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and (c & 0x7F) < 0x60], np.uint8)
    k8 = rng.choice(finite, size=(slots, Hkv, d))
    v8 = rng.choice(np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8), size=(slots, Hkv, d))
    as_bf16 = lambda c: (F8.decode_e4m3(c).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert (A.widen(as_bf16(k8)) == F8.decode_e4m3(k8)).all()
    table = rng.permutation(np.arange(1, 16, dtype=np.int32))[:6].reshape(B, 3)
    q = (rng.normal(0, 0.3, (B * R, Hq, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    mask = [[int(x) for x in rng.integers(0, 1 << W, R)] for _ in range(B)]
    pos = [[p + r for r in range(R)] for p in P]
    args = (table, P, mask, pos, W, Hkv, THETA)
    o8, l8 = A.window_attention(q, k8, v8, *args, page_size=page, kv_fp8=True)
    ob, lb = A.window_attention(q, as_bf16(k8), as_bf16(v8), *args, page_size=page)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)
    o_sw, _ = A.window_attention(q, v8, k8, *args, page_size=page, kv_fp8=True)
    assert not np.allclose(o_sw, o8)


def test_fp8_query_cast():
    """q_fp8: a query whose values are already E4M3 values is left as it is
    (the cast is exact there); any other query moves by at most one E4M3 step
    per element, and so do the scores: the result changes, within that bound
    on the log-sum-exp."""
    from oracle import fp8 as F8
    rng = np.random.default_rng(92)
    B, R, W, Hq, Hkv, d, page = 1, 2, 3, 2, 1, 8, 4
    k = rng.normal(0, 1, (32, Hkv, d))
    v = rng.normal(0, 1, (32, Hkv, d))
    table = np.array([[3, 5, 1]], np.int32)
    args = (k, v, table, [6], [[5, 3]], [[0, 0]], W, Hkv, THETA)
    q8 = F8.decode_e4m3(rng.integers(0, 0x60, (B * R, Hq, d)).astype(np.uint8))
    o1, l1 = A.window_attention(q8, *args, page_size=page, q_rotated=True, q_fp8=True)
    o0, l0 = A.window_attention(q8, *args, page_size=page, q_rotated=True)
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)
    q = rng.normal(0, 1, (B * R, Hq, d))
    o1, l1 = A.window_attention(q, *args, page_size=page, q_rotated=True, q_fp8=True)
    o0, l0 = A.window_attention(q, *args, page_size=page, q_rotated=True)
    assert not np.allclose(l1, l0)
    # |q8 - q| <= 2^-4 |q| elementwise, so each score moves by at most
    # 2^-4 sum_i |q_i k_i| / sqrt(d), and the log-sum-exp by no more
    bound = 2.0 ** -4 * np.abs(q[:, :, None, :] * k[None, :, 0, None, :].transpose(0, 2, 1, 3)).sum(-1).max() \
        / math.sqrt(d) / math.log(2)
    assert np.abs(l1 - l0).max() <= bound


def test_fp8_query_scores_the_prefix_only():
    """q_fp8 casts the query for the prefix keys alone: with no prefix (only
    window keys visible) the cast changes nothing, and with no window key
    visible the result is that of a query cast beforehand. A cast applied to
    the window keys too, or to neither part, fails one of the two."""
    from oracle import fp8 as F8
    rng = np.random.default_rng(93)
    B, R, W, Hq, Hkv, d, page = 1, 3, 4, 4, 2, 16, 4
    k = rng.normal(0, 1, (32, Hkv, d))
    v = rng.normal(0, 1, (32, Hkv, d))
    table = np.array([[3, 5, 1, 6]], np.int32)
    q = rng.normal(0, 1, (B * R, Hq, d))
    # window keys only (P = 0): every row sees some window keys
    args0 = (k, v, table, [0], [[1, 3, 0b1101]], [[0, 0, 0]], W, Hkv, THETA)
    o1, l1 = A.window_attention(q, *args0, page_size=page, q_rotated=True, q_fp8=True)
    o0, l0 = A.window_attention(q, *args0, page_size=page, q_rotated=True)
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)
    # prefix keys only (mask 0): the same as casting the query first
    args1 = (k, v, table, [9], [[0, 0, 0]], [[0, 0, 0]], W, Hkv, THETA)
    q8 = F8.decode_e4m3(F8.encode_e4m3(q))
    o1, l1 = A.window_attention(q, *args1, page_size=page, q_rotated=True, q_fp8=True)
    o0, l0 = A.window_attention(q8, *args1, page_size=page, q_rotated=True)
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)
    o2, l2 = A.window_attention(q, *args1, page_size=page, q_rotated=True)
    assert not np.allclose(l2, l1)
