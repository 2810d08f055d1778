"""Pins for oracle.rope, oracle.attention and oracle.merge.

The attention oracle is checked against a separately written causal
attention (complex-number RoPE, scipy log-sum-exp, one dense score matrix),
which it must reproduce for a chain and, path by path, for every node of a
tree; and against properties of softmax attention that fix the scale, the
head mapping and the visibility rule.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import attention as A
from oracle import merge as M
from oracle import rope as R
from oracle import tree as T

THETA = 5.0e5


def _va(*a, **k):
    """The oracle with the exact rotation (these pins use non-bf16 inputs);
    the bf16 rounding of rotated tensors is pinned on its own below."""
    k.setdefault("rope_out", None)
    return A.verify_attention(*a, **k)


# ----------------------------------------------------------------------------
# an independent causal attention over one sequence
# ----------------------------------------------------------------------------

def rope_complex(x, pos, theta):
    """RoPE as a complex rotation: z_k = x_k + i x_{k+d/2}, z_k * exp(i pos w_k)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    w = np.array([theta ** (-(2.0 * k) / d) for k in range(d // 2)])
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    z = z * np.exp(1j * np.asarray(pos, np.float64)[..., None] * w)
    return np.concatenate([z.real, z.imag], axis=-1)


def causal_attention(q_seq, k_seq, v_seq, n_pre_rotated, theta, Hkv):
    """q_seq [L][Hq][d] (raw), k_seq/v_seq [L][Hkv][d]; the first n_pre_rotated
    keys are already rotated; token t sits at position t. Returns (out, lse2)
    for every query t >= n_pre_rotated: [L - n][Hq][d], [L - n][Hq]."""
    L, Hq, d = q_seq.shape
    g = Hq // Hkv
    pos = np.arange(L)
    k = np.array(k_seq, np.float64)
    k[n_pre_rotated:] = rope_complex(k[n_pre_rotated:], pos[n_pre_rotated:, None], theta)
    q = rope_complex(q_seq, pos[:, None], theta)
    outs, lses = [], []
    for t in range(n_pre_rotated, L):
        o_t, l_t = [], []
        for h in range(Hq):
            s = np.array([np.dot(q[t, h], k[j, h // g]) for j in range(t + 1)]) / math.sqrt(d)
            l = logsumexp(s)
            p = np.exp(s - l)
            o_t.append(p @ v_seq[: t + 1, h // g])
            l_t.append(l / math.log(2.0))
        outs.append(o_t)
        lses.append(l_t)
    return np.array(outs), np.array(lses)


def _case(rng, B, N, Hq, Hkv, d, P, parents, page=4):
    """Small paged inputs (floats, not bf16) with a shuffled page table."""
    need = (P + N + page - 1) // page
    perm = rng.permutation(np.arange(1, B * need + 1))
    table = perm.reshape(B, need)
    slots = (B * need + 1) * page
    q = rng.standard_normal((B * N, Hq, d))
    kn = rng.standard_normal((B * N, Hkv, d))
    vn = rng.standard_normal((B * N, Hkv, d))
    kc = rng.standard_normal((slots, Hkv, d))
    vc = rng.standard_normal((slots, Hkv, d))
    par = np.array([parents] * B)
    return q, kn, vn, kc, vc, table, np.array([P] * B), par


def _prefix_seq(kc, vc, table, b, P, page):
    sl = A.prefix_slots(table[b], P, page)
    return kc[sl], vc[sl]


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 3, 64))
    pos = rng.integers(0, 200000, size=(7, 3))
    assert np.allclose(R.rotate(x, pos, THETA), rope_complex(x, pos, THETA), atol=1e-12)


def test_rope_properties():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert np.allclose(R.rotate(q, 0, THETA), q)
    assert np.isclose(np.linalg.norm(R.rotate(q, 131136, THETA)), np.linalg.norm(q))
    for m, n in [(5, 3), (131136, 131072), (9, 0)]:
        lhs = R.rotate(q, m, THETA) @ R.rotate(k, n, THETA)
        rhs = R.rotate(q, m - n, THETA) @ k           # scores depend on m - n only
        assert np.isclose(lhs, rhs, atol=1e-9)


def test_chain_equals_causal_attention():
    rng = np.random.default_rng(3)
    B, N, Hq, Hkv, d, P, page = 2, 6, 4, 2, 16, 9, 4
    parents = list(range(-1, N - 1))
    q, kn, vn, kc, vc, table, plen, par = _case(rng, B, N, Hq, Hkv, d, P, parents, page)
    out, lse2 = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    for b in range(B):
        kp, vp = _prefix_seq(kc, vc, table, b, P, page)
        qseq = np.concatenate([np.zeros((P, Hq, d)), q[b * N:(b + 1) * N]])
        kseq = np.concatenate([kp, kn[b * N:(b + 1) * N]])
        vseq = np.concatenate([vp, vn[b * N:(b + 1) * N]])
        o_ref, l_ref = causal_attention(qseq, kseq, vseq, P, THETA, Hkv)
        assert np.allclose(out[b * N:(b + 1) * N], o_ref, atol=1e-12)
        assert np.allclose(lse2[b * N:(b + 1) * N], l_ref, atol=1e-12)


@pytest.mark.parametrize("parents", [
    [-1, 0, 0, 1, 2],                      # [root, A, B, C, D]
    [-1, 0, 0, 0, 0, 0],                   # star
    [-1, 0, 1, 2, 0, 1],                   # the DDTree example
    [-1, 0, 0, 1, 2, 3, 4, 5],             # the build-tree test drawing
])
def test_each_node_is_its_own_root_path(parents):
    """Brute force: node v's row equals causal attention over prefix + path(v)."""
    rng = np.random.default_rng(4)
    N = len(parents)
    B, Hq, Hkv, d, P, page = 1, 4, 2, 8, 5, 4
    q, kn, vn, kc, vc, table, plen, par = _case(rng, B, N, Hq, Hkv, d, P, parents, page)
    out, lse2 = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    kp, vp = _prefix_seq(kc, vc, table, 0, P, page)
    for v in range(N):
        path = T.root_path(parents, v)
        qseq = np.concatenate([np.zeros((P, Hq, d)), q[path]])
        kseq = np.concatenate([kp, kn[path]])
        vseq = np.concatenate([vp, vn[path]])
        o_ref, l_ref = causal_attention(qseq, kseq, vseq, P, THETA, Hkv)
        assert np.allclose(out[v], o_ref[-1], atol=1e-12)
        assert np.allclose(lse2[v], l_ref[-1], atol=1e-12)


def test_star_sees_prefix_root_and_itself():
    rng = np.random.default_rng(5)
    N, Hq, Hkv, d, P, page = 5, 2, 1, 8, 7, 4
    parents = [-1, 0, 0, 0, 0]
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, P, parents, page)
    out, _ = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    # changing node 3's K/V changes only row 3
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[3] += 1.0
    vn2[3] -= 2.0
    out2, _ = _va(q, kn2, vn2, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    changed = [v for v in range(N) if not np.array_equal(out[v], out2[v])]
    assert changed == [3]


def test_non_ancestors_are_never_read():
    """NaN in the K/V of every non-ancestor of v leaves row v bit-identical."""
    rng = np.random.default_rng(6)
    parents = [-1, 0, 0, 1, 2, 1, 0]
    N, Hq, Hkv, d, P, page = len(parents), 4, 2, 8, 6, 4
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, P, parents, page)
    out, lse2 = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    for v in range(N):
        anc = set(T.ancestors(parents, v))
        kn2, vn2 = kn.copy(), vn.copy()
        for j in range(N):
            if j not in anc:
                kn2[j] = np.nan
                vn2[j] = np.inf
        o2, l2 = _va(q, kn2, vn2, kc, vc, table, plen, par, Hkv, THETA,
                                    page_size=page, rows=[(0, v)])
        assert np.array_equal(o2[v], out[v]) and np.array_equal(l2[v], lse2[v])


def test_gqa_head_mapping_and_scale():
    """Hq = 2*Hkv: heads 2k and 2k+1 read KV head k; with the scale given
    explicitly as 1/sqrt(d) the default must agree."""
    rng = np.random.default_rng(7)
    parents = [-1, 0, 1]
    N, Hq, Hkv, d, P, page = 3, 4, 2, 16, 4, 4
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, P, parents, page)
    q[:, 1] = q[:, 0]
    q[:, 3] = q[:, 2]
    out, lse2 = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    assert np.array_equal(out[:, 0], out[:, 1]) and np.array_equal(out[:, 2], out[:, 3])
    assert not np.allclose(out[:, 0], out[:, 2])
    out2, _ = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA,
                                 page_size=page, scale=1.0 / math.sqrt(d))
    assert np.array_equal(out, out2)


def test_zero_prefix_root_row_is_its_own_value():
    """P = 0: the root sees only itself, so out = v_root and lse2 = s/ln2."""
    rng = np.random.default_rng(8)
    N, Hq, Hkv, d, page = 3, 2, 1, 8, 4
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, 0, [-1, 0, 0], page)
    out, lse2 = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    for h in range(Hq):
        assert np.allclose(out[0, h], vn[0, 0])
        s = np.dot(q[0, h], kn[0, 0]) / math.sqrt(d)     # both at position 0: no rotation
        assert np.isclose(lse2[0, h], s / math.log(2.0))


def test_softmax_shift_invariance_and_bf16_widening():
    rng = np.random.default_rng(9)
    parents = [-1, 0, 1, 0]
    N, Hq, Hkv, d, P, page = 4, 2, 1, 8, 5, 4
    q, kn, vn, kc, vc, table, plen, par = _case(rng, 1, N, Hq, Hkv, d, P, parents, page)
    out, lse2 = _va(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    # values shifted by a constant vector: outputs shift by the same vector
    c = rng.standard_normal(d)
    out2, lse2b = _va(q, kn, vn + c, kc, vc + c, table, plen, par, Hkv, THETA,
                                     page_size=page)
    assert np.allclose(out2, out + c, atol=1e-12) and np.allclose(lse2b, lse2)
    bits = np.array([0x3F80, 0xC000, 0x0001], np.uint16)        # 1.0, -2.0, smallest subnormal
    assert A.widen(bits).tolist() == [1.0, -2.0, 2.0 ** -133]


def test_merge_scalar_example(golden):
    g = golden("merge_scalar.txt")
    o, l = M.merge_states(np.array(g["O"], float)[:, None], np.log2(np.array(g["Z"], float)))
    assert o[0] == g["merged"][0]
    assert np.isclose(l, np.log2(sum(g["Z"])))


def test_merge_equals_softmax_over_union():
    rng = np.random.default_rng(10)
    s = rng.standard_normal(40) * 3
    v = rng.standard_normal((40, 5))
    parts = [(0, 7), (7, 8), (8, 40)]
    outs, ls = [], []
    for a, b in parts:
        l = logsumexp(s[a:b])
        outs.append(np.exp(s[a:b] - l) @ v[a:b])
        ls.append(l / math.log(2))
    outs.append(np.zeros(5))            # an empty part carries no mass
    ls.append(-np.inf)
    o, l2 = M.merge_states(outs, ls)
    full = logsumexp(s)
    assert np.allclose(o, np.exp(s - full) @ v, atol=1e-13)
    assert np.isclose(l2, full / math.log(2))


def test_round_bf16_against_torch_cast_and_ties():
    """round_bf16 is round-to-nearest-even to 8 significant bits: it agrees with
    torch's float32 -> bfloat16 cast on float32 inputs, keeps bf16 values, and
    sends exact midpoints to the even neighbour."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(20)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(A.round_bf16(x.astype(np.float64)), want)
    assert A.round_bf16(np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -3.0])).tolist() == \
        [1.0, 1.0, 1.0 + 2.0 ** -6, -3.0]


def test_bf16_storage_of_rotated_tensors():
    """With rope_out='bf16' the oracle equals the exact-rotation oracle fed
    with rotated-then-rounded tensors (window keys rounded at their positions,
    queries at theirs): the chain case against the causal reference."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    B, N, Hq, Hkv, d, P, page = 1, 5, 4, 2, 16, 7, 4
    parents = list(range(-1, N - 1))
    q, kn, vn, kc, vc, table, plen, par = _case(rng, B, N, Hq, Hkv, d, P, parents, page)
    out, lse2 = A.verify_attention(q, kn, vn, kc, vc, table, plen, par, Hkv, THETA, page_size=page)
    pos = P + np.arange(N)

    def rounded(x, p):
        r = rope_complex(x, p[:, None], THETA).astype(np.float32)
        return torch.from_numpy(r).to(torch.bfloat16).to(torch.float64).numpy()
    q_r, k_r = rounded(q, pos), rounded(kn, pos)
    kp, vp = _prefix_seq(kc, vc, table, 0, P, page)
    kseq = np.concatenate([kp, k_r])
    vseq = np.concatenate([vp, vn])
    # causal attention with already-rotated keys and queries (n_pre_rotated = everything)
    L = P + N
    outs, lses = [], []
    for t in range(P, L):
        o_t, l_t = [], []
        for h in range(Hq):
            s = kseq[: t + 1, h // (Hq // Hkv)] @ q_r[t - P, h] / math.sqrt(d)
            l = logsumexp(s)
            o_t.append(np.exp(s - l) @ vseq[: t + 1, h // (Hq // Hkv)])
            l_t.append(l / math.log(2))
        outs.append(o_t)
        lses.append(l_t)
    # the exact-rotation outputs differ by the rounding; the bf16 ones match
    assert np.allclose(out, np.array(outs), atol=1e-6) and np.allclose(lse2, np.array(lses), atol=1e-6)
