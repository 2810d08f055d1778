"""Oracle: tree-verify attention, computed literally per root path in fp64.

Test infrastructure only (see the package docstring).

Definition followed ([AK] section one, "Target Verify" identity; [MI] "Here is
the problem trees solve"): the verify row of node v must equal the target's
attention over the committed prefix followed by v's own root path,
L(v) = Target(prefix + path(root -> v)).

For request b with committed prefix length P (= vc), node v with root path
u_0 = 0, ..., u_D = v, and query head h reading KV head h // (Hq / Hkv):

  keys   = [K_cache(b, p) for p < P] ++ [RoPE(k_new[u_t], P + t) for t = 0..D]
  values = [V_cache(b, p) for p < P] ++ [v_new[u_t]                for t = 0..D]
  q      = RoPE(q_raw[v, h], P + D)
  s      = (q . keys) * scale,         scale = 1/sqrt(d) unless given
  out    = softmax(s) . values
  lse2   = ln(sum exp(s)) / ln 2       (base-2 log-sum-exp, [TS] "One tree attention")

The prefix keys in the cache are already rotated (their positions are p < P).
Window node u_t sits at logical position P + t because its depth is t
([TS] "Position follows depth"); slot follows node index, so the oracle takes
window K/V from k_new/v_new by node index and never reads the mask, the
positions array or the cache's window slots.

Readings taken where the pages are silent: scale 1/sqrt(d); query head h reads
KV head h // (Hq/Hkv); RoPE is the rotate-half form (oracle.rope).

Precision of the rotated tensors: the paged K/V cache is bf16, and a window
node's key enters attention as its slot holds it ([TS] "Position follows
depth, slot follows node index": node i's rotated K is written to its slot),
i.e. RoPE(k_new) rounded to bf16. The query reaches attention in the model
dtype ([TS] "One tree attention", FP8 paragraph: the window kernel takes the
unquantized query), i.e. RoPE(q) rounded to bf16. ``rope_out="bf16"`` (the
default) applies both roundings (round to nearest, ties to even, from the
exact fp64 rotation); ``rope_out=None`` keeps the exact rotation. Everything
after that is fp64.

The prefix scores of many nodes are formed with one matrix product per KV
head (the same dot products, batched); each node's softmax is then taken over
its own concatenated key list.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np

from . import rope
from .tree import root_path

LN2 = math.log(2.0)


def widen(a) -> np.ndarray:
    """bf16 bits (uint16) -> fp64 exactly; float arrays -> fp64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (8 significant bits, ties
    to even), returned as fp64. Finite normal-range inputs only (as here)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def prefix_slots(page_table_row, P: int, page_size: int) -> np.ndarray:
    pos = np.arange(P, dtype=np.int64)
    return np.asarray(page_table_row, dtype=np.int64)[pos // page_size] * page_size + pos % page_size


def verify_attention(q, k_new, v_new, k_cache, v_cache, page_table, prefix_len, parents,
                     Hkv: int, theta: float, page_size: int = 64, scale: Optional[float] = None,
                     rows: Optional[Iterable] = None, q_rotated: bool = False,
                     rope_out: Optional[str] = "bf16", max_chunk_elems: int = 1 << 24):
    """Returns (out [B*N][Hq][d] fp64, lse2 [B*N][Hq] fp64).

    q: [B*N][Hq][d]; k_new, v_new: [B*N][Hkv][d]; k_cache, v_cache:
    [slots][Hkv][d] (bf16 bits or floats); page_table int [B][max_pages];
    prefix_len int [B]; parents int [B][N]. ``rows`` restricts the work to the
    given (b, v) pairs; the other rows are NaN. ``q_rotated`` skips the query
    rotation (the caller passes already-rotated queries). ``rope_out`` is the
    storage precision of the rotated query and window keys ("bf16" or None).
    """
    rnd = round_bf16 if rope_out == "bf16" else (lambda a: a)
    parents = np.asarray(parents)
    B, N = parents.shape
    q = np.asarray(q)
    Hq, d = q.shape[1], q.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.full((B * N, Hq, d), np.nan)
    lse2 = np.full((B * N, Hq), np.nan)
    if rows is None:
        want = {b: list(range(N)) for b in range(B)}
    else:
        want = {}
        for b, v in rows:
            want.setdefault(int(b), []).append(int(v))

    for b, nodes in sorted(want.items()):
        P = int(prefix_len[b])
        slots = prefix_slots(page_table[b], P, page_size)
        Kp = np.ascontiguousarray(widen(np.asarray(k_cache)[slots]).transpose(1, 0, 2))  # [Hkv][P][d]
        Vp = np.ascontiguousarray(widen(np.asarray(v_cache)[slots]).transpose(1, 0, 2))

        # per node: its path, rotated query, rotated window keys
        info = []
        for v in nodes:
            path = root_path(parents[b], v)
            D = len(path) - 1
            rows_bn = [b * N + u for u in path]
            kw = rnd(rope.rotate(widen(np.asarray(k_new)[rows_bn]), P + np.arange(D + 1)[:, None], theta))
            vw = widen(np.asarray(v_new)[rows_bn])                      # [D+1][Hkv][d]
            qv = widen(q[b * N + v])
            if not q_rotated:
                qv = rnd(rope.rotate(qv, P + D, theta))                 # [Hq][d]
            info.append((v, qv, kw, vw))

        chunk = max(1, max_chunk_elems // max(1, P * g))
        for c0 in range(0, len(info), chunk):
            part = info[c0: c0 + chunk]
            for kv in range(Hkv):
                hs = slice(kv * g, (kv + 1) * g)
                Q = np.concatenate([qv[hs] for _, qv, _, _ in part], axis=0)   # [c*g][d]
                S_pre = (Q @ Kp[kv].T) * scale if P > 0 else np.zeros((Q.shape[0], 0))
                for n, (v, qv, kw, vw) in enumerate(part):
                    s_pre = S_pre[n * g:(n + 1) * g]                        # [g][P]
                    s_win = (qv[hs] @ kw[:, kv].T) * scale                  # [g][D+1]
                    s = np.concatenate([s_pre, s_win], axis=1)              # the node's key list
                    m = s.max(axis=1, keepdims=True)
                    e = np.exp(s - m)
                    Z = e.sum(axis=1)
                    o = e[:, :P] @ Vp[kv] + e[:, P:] @ vw[:, kv]
                    out[b * N + v, hs] = o / Z[:, None]
                    lse2[b * N + v, hs] = (m[:, 0] + np.log(Z)) / LN2
    return out, lse2


def prefix_query(qv, q_fp8: bool):
    """The query the prefix keys are scored against: under an FP8 cache the
    decode's query cast to E4M3 ([TS] "One tree attention", FP8 paragraph)."""
    if not q_fp8:
        return qv
    from .fp8 import decode_e4m3, encode_e4m3
    return decode_e4m3(encode_e4m3(qv))


def window_query(qv, q_fp8: bool):
    """The query the window keys are scored against: the unquantized one,
    under an FP8 cache too (the same paragraph: the window kernel takes the
    unquantized query)."""
    return qv


def window_attention(q, k_cache, v_cache, page_table, prefix_len, mask, positions, W: int, Hkv: int,
                     theta: float, page_size: int = 64, scale: Optional[float] = None,
                     q_rotated: bool = False, rope_out: Optional[str] = "bf16", kv_fp8: bool = False,
                     q_fp8: bool = False):
    """Attention of R query rows per request over the committed prefix plus
    a masked window of W keys, all read from the paged cache.

    Definition followed ([TS] "One tree attention": every row sees the
    committed prefix, and the 64-bit ancestor mask applies only to the last
    W keys; verify runs with R = W = N, draft lanes with R = K rows over the
    (S - 1) * K-key lane window; [TS] "Draft lanes write the draft cache like
    any draft step": every lane row sees the accepted frontier and, inside the
    window, only its ancestors' slots, the lane mask):

      keys(b, r) = [K_cache(b, p) for p < P]
                   ++ [K_cache(b, P + j) for j < W with bit j of mask[b][r] set]
      values     = the same positions of V_cache
      q          = RoPE(q_raw[b*R + r, h], positions[b][r]), rounded as in
                   verify_attention (``rope_out``)
      out, lse2  = softmax over the keys (scale 1/sqrt(d)), base-2 LSE

    The window keys are taken as the cache holds them (already rotated by the
    step that wrote them); the oracle builds each row's key list itself and
    never reads a path. Shapes: q [B*R][Hq][d]; k_cache, v_cache
    [slots][Hkv][d]; page_table [B][max_pages]; prefix_len [B]; mask [B][R]
    (uint64 or Python ints); positions [B][R]. Returns (out [B*R][Hq][d],
    lse2 [B*R][Hq]), fp64.

    ``kv_fp8``: the caches hold E4M3 bytes, read as the values they encode
    (oracle.fp8.decode_e4m3; [TS] "One tree attention", FP8 paragraph: the
    cache is unscaled and its K/V are widened after loading). ``q_fp8``: the
    prefix keys are scored against the query (rotated and rounded as above)
    cast to E4M3 (oracle.fp8.encode_e4m3), the window keys against the query
    as it is (the same paragraph: the decode over the committed prefix takes
    the query cast to FP8, the window kernel the unquantized query).
    """
    rnd = round_bf16 if rope_out == "bf16" else (lambda a: a)
    if kv_fp8:
        from .fp8 import decode_e4m3
    load = decode_e4m3 if kv_fp8 else widen
    q = np.asarray(q)
    B = len(prefix_len)
    R = q.shape[0] // B
    Hq, d = q.shape[1], q.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kc, vc = np.asarray(k_cache), np.asarray(v_cache)
    out = np.zeros((B * R, Hq, d))
    lse2 = np.zeros((B * R, Hq))
    for b in range(B):
        P = int(prefix_len[b])
        pt = np.asarray(page_table[b], dtype=np.int64)
        slots_all = prefix_slots(pt, P + W, page_size)
        Kp = load(kc[slots_all[:P]]).transpose(1, 0, 2)                # [Hkv][P][d]
        Vp = load(vc[slots_all[:P]]).transpose(1, 0, 2)
        for r in range(R):
            bits = int(mask[b][r])
            win = [j for j in range(W) if (bits >> j) & 1]
            Kw = load(kc[slots_all[[P + j for j in win]]]).transpose(1, 0, 2) if win else np.zeros((Hkv, 0, d))
            Vw = load(vc[slots_all[[P + j for j in win]]]).transpose(1, 0, 2) if win else np.zeros((Hkv, 0, d))
            qv = widen(q[b * R + r])
            if not q_rotated:
                qv = rnd(rope.rotate(qv, int(positions[b][r]), theta))
            qp, qw = prefix_query(qv, q_fp8), window_query(qv, q_fp8)
            for kv in range(Hkv):
                hs = slice(kv * g, (kv + 1) * g)
                vals = np.concatenate([Vp[kv], Vw[kv]], axis=0)         # [P + |win|][d]
                if vals.shape[0] == 0:                                   # nothing visible: 0 and -inf
                    out[b * R + r, hs] = 0.0
                    lse2[b * R + r, hs] = -np.inf
                    continue
                s = np.concatenate([qp[hs] @ Kp[kv].T, qw[hs] @ Kw[kv].T], axis=1) * scale  # [g][keys]
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                Z = e.sum(axis=1)
                out[b * R + r, hs] = (e @ vals) / Z[:, None]
                lse2[b * R + r, hs] = (m[:, 0] + np.log(Z)) / LN2
    return out, lse2
