"""Seeded synthetic inputs for the target-verify step of draft-tree speculation.

This module is shared by the tests, ``bench.py`` and the oracle's callers. It
draws random numbers and lays them out; it holds none of the verify step's own
arithmetic (no mask, no attention, no walk, no compaction). Tree *construction*
(the drafter's side: candidate scoring, selection and depth-first numbering)
lives here because it only produces the ``parents``/``depth`` inputs.

Workloads (each named by what it is, with its sizes):

* ``tiny_p128_n5``       B=1, Hq=4, Hkv=1, d=64, P=128, the fixed tree
  [root, A, B, C, D] with parents [-1, 0, 0, 1, 2]; contiguous KV.
* ``llama8b_p4096_n8``   B=8, Hq=32, Hkv=8, d=128, P=4096, N=8 from a full
  topk=2, depth-3 expansion (best 7 of 14 plus the root); paged KV.
* ``eagle2_p8192_n64``   B=32, Hq=32, Hkv=8, d=128, P=8192, N=64 from an
  EAGLE-2 beam (topk=8, 6 steps, pool 328); paged KV.
* ``longctx_p131072_n64`` B=4, Hq=64, Hkv=8, d=128, ragged
  P=131072/98304/65536/32768, N=64 EAGLE-2 trees as above.
* ``highconc_b128_n16``  B=128, Hq=32, Hkv=8, d=128, P ~ U{512..4096}, N=16
  from an EAGLE-2 beam (topk=4, 4 steps, pool 52), plus 32 layers of fp8
  K/V buffers and bf16 hidden rows (dim 4096) for compaction.

Random streams: ``PCG64(SeedSequence(20261202 + index))`` spawns one child
stream per tensor in a fixed order, so any one tensor can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

SEED_BASE = 20261202
PAGE_SIZE = 64
ROPE_THETA = 5.0e5

# Child-stream order; never reorder (it would change every stored value).
_STREAMS = ("tree", "tokens", "q", "k_cache", "v_cache", "k_new", "v_new",
            "pages", "hidden", "fp8", "prefix", "logits")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    d: int
    N: int
    prefix: Sequence[int] | str       # explicit per-request P, or "uniform512_4096"
    tree: str                         # "fixed_root_abcd" | "full" | "eagle2"
    topk: int = 0
    steps: int = 0
    vocab: int = 128256
    token_rule: str = "copy_parent_argmax_0.7"
    contiguous: bool = False
    hidden_dim: int = 4096
    fp8_layers: int = 0               # layers of fp8 K/V for compaction (K and V each)
    rope_theta: float = ROPE_THETA
    page_size: int = PAGE_SIZE

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_p128_n5", 0, B=1, Hq=4, Hkv=1, d=64, N=5, prefix=[128],
                 tree="fixed_root_abcd", vocab=1000, token_rule="copy_parent_argmax_0.5",
                 contiguous=True, hidden_dim=256),
        Workload("llama8b_p4096_n8", 1, B=8, Hq=32, Hkv=8, d=128, N=8, prefix=[4096] * 8,
                 tree="full", topk=2, steps=3),
        Workload("eagle2_p8192_n64", 2, B=32, Hq=32, Hkv=8, d=128, N=64, prefix=[8192] * 32,
                 tree="eagle2", topk=8, steps=6),
        Workload("longctx_p131072_n64", 3, B=4, Hq=64, Hkv=8, d=128, N=64,
                 prefix=[131072, 98304, 65536, 32768], tree="eagle2", topk=8, steps=6,
                 hidden_dim=8192),
        Workload("highconc_b128_n16", 4, B=128, Hq=32, Hkv=8, d=128, N=16,
                 prefix="uniform512_4096", tree="eagle2", topk=4, steps=4, fp8_layers=32),
    ]
}


def workload_by_index(i: int) -> Workload:
    for w in WORKLOADS.values():
        if w.index == i:
            return w
    raise KeyError(i)


def streams(index: int) -> dict:
    """One independent generator per named tensor, in a fixed spawn order."""
    children = np.random.SeedSequence(SEED_BASE + index).spawn(len(_STREAMS))
    return {name: np.random.Generator(np.random.PCG64(ss)) for name, ss in zip(_STREAMS, children)}


# ----------------------------------------------------------------------------
# bf16 helpers (storage only: round-to-nearest-even of fp32 draws)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the raw uint16 bits.
    Finite inputs cannot overflow the uint32 sum (the largest is 0xFF7FFFFF)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    step = 1 << 24
    for o in range(0, flat.size, step):
        u = flat[o:o + step].view(np.uint32)
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        out[o:o + step] = r.astype(np.uint16)
    nan = np.isnan(flat)
    if nan.any():
        out[nan] = 0x7FC0
    return out.reshape(x.shape)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) drawn in fp32 and rounded to bf16; returned as uint16 bits."""
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def normal_e4m3(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1)-shaped E4M3 bytes (storage only, no rounding): the sign, the
    exponent (rebiased from 127 to 7) and the three leading mantissa bits of
    an fp32 draw. Draws below 2^-6 in magnitude store zero; none of an N(0,1)
    draw reaches the top binade [256, 512), so no NaN code appears."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)
    step = 1 << 24
    for o in range(0, n, step):
        u = rng.standard_normal(size=min(step, n - o), dtype=np.float32).view(np.uint32)
        e = ((u >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int32) - 120
        m = ((u >> np.uint32(20)) & np.uint32(7)).astype(np.int32)
        code = np.where(e < 1, 0, (np.minimum(e, 15) << 3) | m)
        code = np.minimum(code, 0x7E)
        out[o:o + step] = (code | ((u >> np.uint32(31)).astype(np.int32) << 7)).astype(np.uint8)
    return out.reshape(shape)


def fp8_kv_cache(index: int, num_slots: int, Hkv: int, d: int):
    """E4M3 K and V caches [num_slots][Hkv][d] from a workload's k_cache and
    v_cache streams (every key taken as already rotated at its position)."""
    s = streams(index)
    return normal_e4m3(s["k_cache"], (num_slots, Hkv, d)), normal_e4m3(s["v_cache"], (num_slots, Hkv, d))


# ----------------------------------------------------------------------------
# Draft trees (drafter side; produces the verify step's parents/depth inputs)
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class _Cand:
    cid: int
    parent: int      # candidate id of the parent, -1 = the root
    score: float     # cumulative log-probability (<= parent's)
    depth: int


def _sorted_child_logp(rng: np.random.Generator, topk: int) -> np.ndarray:
    p = np.sort(rng.dirichlet(0.5 * np.ones(topk)))[::-1]
    with np.errstate(divide="ignore"):
        lp = np.log(p)
    return np.minimum(lp, 0.0)  # a child never outscores its parent


def _rank_key(c: _Cand):
    s = c.score
    if np.isnan(s):
        s = -np.inf
    return (-s, c.depth, c.cid)


def _select_and_number(cands: List[_Cand], n_nodes: int):
    """Keep the best n_nodes-1 candidates (score desc, depth asc, id asc), then
    number the kept tree depth-first with each node's best child first."""
    ranked = sorted(cands, key=_rank_key)
    kept = ranked[: n_nodes - 1]
    kept_ids = {c.cid for c in kept}
    for c in kept:
        if c.parent != -1 and c.parent not in kept_ids:
            raise AssertionError("selected candidate set is not ancestor-closed")
    children = {-1: []}
    for c in kept:
        children.setdefault(c.cid, [])
    for c in sorted(kept, key=_rank_key):
        children[c.parent].append(c)
    order = []                       # DFS preorder; the root is node 0
    parents = [-1]
    depth = [0]
    node_of = {-1: 0}

    def visit(cid):                  # preorder, best child first
        for ch in children[cid]:
            node_of[ch.cid] = len(parents)
            parents.append(node_of[cid])
            depth.append(ch.depth)
            order.append(ch.cid)
            visit(ch.cid)
    visit(-1)
    return np.array(parents, np.int32), np.array(depth, np.int32), order


def tree_full_expansion(rng: np.random.Generator, topk: int, steps: int, n_nodes: int):
    """Every node up to depth `steps` expands `topk` children; keep the best n_nodes-1."""
    cands: List[_Cand] = []
    frontier = [(-1, 0.0, 0)]
    for _ in range(steps):
        nxt = []
        for pid, pscore, pdepth in frontier:
            for lp in _sorted_child_logp(rng, topk):
                c = _Cand(len(cands), pid, pscore + lp, pdepth + 1)
                cands.append(c)
                nxt.append((c.cid, c.score, c.depth))
        frontier = nxt
    return _select_and_number(cands, n_nodes)


def tree_eagle2(rng: np.random.Generator, topk: int, steps: int, n_nodes: int):
    """EAGLE-2 style beam: the root expands topk children; at each later step the
    current topk survivors each expand topk children and the global best topk of
    those survive. Pool = topk + (steps-1)*topk^2 candidates; keep n_nodes-1."""
    cands: List[_Cand] = []
    frontier = []
    for lp in _sorted_child_logp(rng, topk):
        c = _Cand(len(cands), -1, float(lp), 1)
        cands.append(c)
        frontier.append(c)
    for _ in range(steps - 1):
        new = []
        for f in frontier:
            for lp in _sorted_child_logp(rng, topk):
                c = _Cand(len(cands), f.cid, f.score + float(lp), f.depth + 1)
                cands.append(c)
                new.append(c)
        frontier = sorted(new, key=_rank_key)[:topk]
    return _select_and_number(cands, n_nodes)


FIXED_ROOT_ABCD = (np.array([-1, 0, 0, 1, 2], np.int32), np.array([0, 1, 1, 2, 2], np.int32))


def make_trees(w: Workload, rng: np.random.Generator):
    parents = np.zeros((w.B, w.N), np.int32)
    depth = np.zeros((w.B, w.N), np.int32)
    for b in range(w.B):
        if w.tree == "fixed_root_abcd":
            p, dp = FIXED_ROOT_ABCD
        elif w.tree == "full":
            p, dp, _ = tree_full_expansion(rng, w.topk, w.steps, w.N)
        elif w.tree == "eagle2":
            p, dp, _ = tree_eagle2(rng, w.topk, w.steps, w.N)
        else:
            raise ValueError(w.tree)
        parents[b], depth[b] = p, dp
    return parents, depth


def chain_tree(n: int):
    return np.arange(-1, n - 1, dtype=np.int32), np.arange(n, dtype=np.int32)


def star_tree(n: int):
    p = np.zeros(n, np.int32)
    p[0] = -1
    dp = np.ones(n, np.int32)
    dp[0] = 0
    return p, dp


def depth_of(parents: np.ndarray) -> np.ndarray:
    """Depth from parents (parents[i] < i). Used to build inputs, not to check them."""
    dp = np.zeros(len(parents), np.int32)
    for i in range(1, len(parents)):
        dp[i] = dp[parents[i]] + 1
    return dp


# ----------------------------------------------------------------------------
# Tokens
# ----------------------------------------------------------------------------

def make_tokens(w: Workload, parents: np.ndarray, rng: np.random.Generator):
    """target_argmax: the argmax of iid N(0,1) target logits is uniform over the
    vocabulary, so it is drawn uniformly. draft: each child copies its parent's
    target argmax with probability p (0.5 or 0.7), else a uniform token."""
    p_copy = 0.5 if w.token_rule.endswith("0.5") else 0.7
    B, N = parents.shape
    target_argmax = rng.integers(0, w.vocab, size=(B, N), dtype=np.int64).astype(np.int32)
    draft = rng.integers(0, w.vocab, size=(B, N), dtype=np.int64).astype(np.int32)
    copy = rng.random(size=(B, N)) < p_copy
    for b in range(B):
        for i in range(1, N):
            if copy[b, i]:
                draft[b, i] = target_argmax[b, parents[b, i]]
    return draft, target_argmax


# ----------------------------------------------------------------------------
# Paged KV layout
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class PagedLayout:
    prefix_len: np.ndarray    # int32 [B]   (= vc, the committed prefix)
    page_table: np.ndarray    # int32 [B][max_pages]; unused entries point at page 0
    num_pages: int            # pool size including the reserved page 0
    num_slots: int
    write_locations: np.ndarray  # int64 [B*N]: slot of window node i of request b
    page_size: int = PAGE_SIZE

    def slot(self, b: int, pos: int) -> int:
        ps = self.page_size
        return int(self.page_table[b, pos // ps]) * ps + pos % ps


def make_prefix_lens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if isinstance(w.prefix, str):
        assert w.prefix == "uniform512_4096"
        return rng.integers(512, 4097, size=w.B, dtype=np.int64).astype(np.int32)
    return np.array(w.prefix, np.int32)


def make_layout(w: Workload, prefix_len: np.ndarray, rng: np.random.Generator,
                extra_pages: int = 0) -> PagedLayout:
    """Each request owns ceil((P_b + N)/64) pages: its prefix, then the verify
    window at logical positions P_b .. P_b+N-1. Physical page 0 is reserved (a
    dummy slot resolves there); the others are a seeded random permutation of
    the pool, or in order for a contiguous layout."""
    B, N, ps = w.B, w.N, w.page_size
    need = [(int(p) + N + ps - 1) // ps for p in prefix_len]
    total = sum(need) + extra_pages
    phys = np.arange(1, total + 1, dtype=np.int64)
    if not w.contiguous:
        phys = rng.permutation(phys)
    max_pages = max(need)
    table = np.zeros((B, max_pages), np.int32)
    o = 0
    for b in range(B):
        table[b, : need[b]] = phys[o: o + need[b]]
        o += need[b]
    num_pages = total + 1
    wl = np.zeros(B * N, np.int64)
    lay = PagedLayout(prefix_len.astype(np.int32), table, num_pages, num_pages * ps, wl, ps)
    for b in range(B):
        for i in range(N):
            wl[b * N + i] = lay.slot(b, int(prefix_len[b]) + i)
    return lay


# ----------------------------------------------------------------------------
# One full set of inputs for a workload
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class VerifyInputs:
    w: Workload
    parents: np.ndarray        # int32 [B][N]
    depth: np.ndarray          # int32 [B][N]
    draft: np.ndarray          # int32 [B][N]
    target_argmax: np.ndarray  # int32 [B][N]
    layout: PagedLayout
    q: np.ndarray              # bf16 bits [B*N][Hq][d] (not rotated)
    k_new: np.ndarray          # bf16 bits [B*N][Hkv][d] (not rotated)
    v_new: np.ndarray          # bf16 bits [B*N][Hkv][d]
    k_cache: np.ndarray        # bf16 bits [num_slots][Hkv][d] (prefix keys already rotated)
    v_cache: np.ndarray        # bf16 bits [num_slots][Hkv][d]
    hidden: Optional[np.ndarray] = None  # bf16 bits [B*N][hidden_dim]

    @property
    def vc(self) -> np.ndarray:
        return self.layout.prefix_len


def make_inputs(w: Workload, with_cache: bool = True, with_hidden: bool = True,
                prefix_override: Optional[Sequence[int]] = None,
                trees=None) -> VerifyInputs:
    s = streams(w.index)
    if trees is None:
        parents, depth = make_trees(w, s["tree"])
    else:
        parents, depth = trees
    draft, argmax = make_tokens(w, parents, s["tokens"])
    plen = make_prefix_lens(w, s["prefix"]) if prefix_override is None else np.array(prefix_override, np.int32)
    lay = make_layout(w, plen, s["pages"])
    BN = w.B * w.N
    q = normal_bf16(s["q"], (BN, w.Hq, w.d))
    k_new = normal_bf16(s["k_new"], (BN, w.Hkv, w.d))
    v_new = normal_bf16(s["v_new"], (BN, w.Hkv, w.d))
    if with_cache:
        k_cache = normal_bf16(s["k_cache"], (lay.num_slots, w.Hkv, w.d))
        v_cache = normal_bf16(s["v_cache"], (lay.num_slots, w.Hkv, w.d))
    else:
        k_cache = v_cache = None
    hidden = normal_bf16(s["hidden"], (BN, w.hidden_dim)) if with_hidden else None
    return VerifyInputs(w, parents, depth, draft, argmax, lay, q, k_new, v_new, k_cache, v_cache, hidden)


# A logit no N(0,1) draw comes near (P(N(0,1) > 20) is about 3e-89).
PLANTED_LOGIT = 20.0


def target_logits(w: Workload, target_argmax: np.ndarray) -> np.ndarray:
    """fp32 target logits [B*N][vocab] for the verify rows: iid N(0,1) draws,
    with each row's entry at that row's drawn target token set to
    PLANTED_LOGIT, so the target tokens drawn by make_tokens (and the drafts
    made from them) are the rows' argmax by construction."""
    rng = streams(w.index)["logits"]
    rows = w.B * w.N
    x = rng.standard_normal((rows, w.vocab), dtype=np.float32)
    x[np.arange(rows), np.asarray(target_argmax).reshape(-1)] = PLANTED_LOGIT
    return x


# ----------------------------------------------------------------------------
# Draft-lane attention inputs (drafter side: lane ancestry and lane masks)
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LaneWorkload:
    """K lane rows per request at drafting step `step` (1 <= step <= S - 1;
    0 means the last, S - 1) over the (S - 1) * K-key lane window of the
    draft cache; window key (s - 1) * K + r is the key lane r wrote at step s."""
    name: str
    index: int
    B: int
    K: int
    S: int
    Hq: int
    Hkv: int
    d: int
    prefix: Sequence[int]
    step: int = 0
    page_size: int = PAGE_SIZE
    rope_theta: float = ROPE_THETA

    @property
    def W(self) -> int:
        return (self.S - 1) * self.K

    @property
    def R(self) -> int:
        return self.K


LANE_WORKLOADS = {
    # the EAGLE-2 batch's drafting: topk 8 lanes, 6 drafting steps (S = 7), the
    # draft head with the target's attention shape, over its 8192-token frontier
    "lanes_eagle2_p8192_k8_s7": LaneWorkload("lanes_eagle2_p8192_k8_s7", 10, B=32, K=8, S=7, Hq=32, Hkv=8, d=128,
                                             prefix=[8192] * 32),
}


@dataclasses.dataclass
class LaneInputs:
    lw: LaneWorkload
    mask: np.ndarray        # uint64 [B][K]: bit j = window key j is an ancestor of (or is) the lane's token
    positions: np.ndarray   # int32 [B][K]: the lane tokens' positions
    layout: PagedLayout
    q: np.ndarray           # bf16 bits [B*K][Hq][d] (not rotated)
    k_cache: np.ndarray     # bf16 bits, or E4M3 bytes, [num_slots][Hkv][d] (all keys already rotated)
    v_cache: np.ndarray

    @property
    def prefix_len(self) -> np.ndarray:
        return self.layout.prefix_len


def make_lane_inputs(lw: LaneWorkload, kv_fp8: bool = False) -> LaneInputs:
    """Seeded lane inputs. The drafter's beam keeps K lanes per step; lane r of
    step s >= 2 descends from a lane of step s - 1 drawn uniformly (several
    lanes may share a parent), and a lane's mask holds its own key's bit and
    its ancestors' (one per earlier step). kv_fp8: the caches are E4M3 bytes
    (normal_e4m3) instead of bf16 bits."""
    s = streams(lw.index)
    B, K, W = lw.B, lw.K, lw.W
    step = lw.step or lw.S - 1
    rng = s["tree"]
    masks = np.zeros((B, K), np.uint64)
    for b in range(B):
        prev = [0] * K
        for st in range(1, step + 1):
            cur = []
            for r in range(K):
                m = 1 << ((st - 1) * K + r)
                if st >= 2:
                    m |= prev[int(rng.integers(0, K))]
                cur.append(m)
            prev = cur
        masks[b] = np.array(prev, dtype=np.uint64)
    plen = np.array(lw.prefix, np.int32)
    w = Workload(lw.name, lw.index, B=B, Hq=lw.Hq, Hkv=lw.Hkv, d=lw.d, N=W, prefix=list(lw.prefix), tree="lanes",
                 page_size=lw.page_size, rope_theta=lw.rope_theta)
    lay = make_layout(w, plen, s["pages"])
    positions = (plen[:, None] + step - 1 + np.zeros((1, K), np.int32)).astype(np.int32)
    q = normal_bf16(s["q"], (B * K, lw.Hq, lw.d))
    draw = normal_e4m3 if kv_fp8 else normal_bf16
    k_cache = draw(s["k_cache"], (lay.num_slots, lw.Hkv, lw.d))
    v_cache = draw(s["v_cache"], (lay.num_slots, lw.Hkv, lw.d))
    return LaneInputs(lw, masks, positions, lay, q, k_cache, v_cache)


def fp8_window_rows(w: Workload, n_buffers: int, row_bytes: int) -> np.ndarray:
    """Random bytes for the window slots of each fp8 K/V buffer: uint8 [L][B*N][row_bytes]."""
    rng = streams(w.index)["fp8"]
    return rng.integers(0, 256, size=(n_buffers, w.B * w.N, row_bytes), dtype=np.uint8)
