"""Oracle: sampled tree verification, Gumbel-max draws keyed by position.

Test infrastructure only (see the package docstring).

Source: [TS] "Sampled verify keys noise by position": a verify row's target
token is drawn by Gumbel-max keyed by (seed, position); for a tree the key is
the position the node predicts, vc + depth + 1 (vc the pre-forward frontier),
never the row, so every node samples with its request's parameters and the
token accepted at each position is the one plain decoding samples there.
Acceptance is the greedy tree walk over those draws (a child is accepted when
it equals its parent's draw).

The draw of row (b, i) is  argmax_v  x_v * (1/T_b) + G(seed_b, pos, v),
pos = vc_b + depth[b][i] + 1, with NumPy's argmax rules (oracle.argmax).
T_b <= 0 (or not finite) selects the plain argmax, no noise.

Readings taken where the page is silent (the noise generator, its key and
counter layout, the float arithmetic) - every one is fixed so that the
arithmetic, all in float32 with one IEEE rounding per operation and no fused
multiply-add, is reproducible bit for bit:

* Random words: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
  numbers: as easy as 1, 2, 3", SC 2011): key (seed low word, seed high word),
  counter (v // 4, pos, 0, 0); word v % 4 of the output block belongs to
  vocabulary entry v.
* Uniform: u = (2 * (word >> 9) + 1) * 2^-24, exact in float32, in
  [2^-24, 1 - 2^-24].
* Gumbel: G = -ln(-ln(u)), with ln computed by ``log_f32`` below.
* Scaled logit: x * (1/T) with 1/T one float32 division, then + G.
"""
from __future__ import annotations

import numpy as np

from . import argmax as _argmax
from . import walk as _walk

_M0, _M1 = 0xD2511F53, 0xCD9E8D57          # Philox4x32 round multipliers
_W0, _W1 = 0x9E3779B9, 0xBB67AE85          # Philox4x32 key increments
_MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """ctr: uint array [..., 4]; key: uint array [..., 2] (broadcastable).
    Returns the four output words, uint32 [..., 4]."""
    c = [np.asarray(ctr, np.uint64)[..., i] & _MASK for i in range(4)]
    k0 = np.asarray(key, np.uint64)[..., 0] & _MASK
    k1 = np.asarray(key, np.uint64)[..., 1] & _MASK
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = np.uint64(_M0) * c[0]
        p1 = np.uint64(_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack(c, axis=-1).astype(np.uint32)


_F = np.float32
_LN2 = _F(0.6931471805599453)       # ln 2 rounded to float32
_SQRT2 = _F(1.4142135623730951)
_C = [_F(1.0), _F(1.0 / 3.0), _F(1.0 / 5.0), _F(1.0 / 7.0), _F(1.0 / 9.0)]


def log_f32(x):
    """Natural log of positive normal float32 values, as this exact float32
    sequence (each operation rounded once, to nearest even):
        x = m * 2^e with m in [1, 2); if m > sqrt(2): m = m / 2, e = e + 1
        s = (m - 1) / (m + 1);  t = s * s
        p = (((t/9 + 1/7) t + 1/5) t + 1/3) t + 1        (coefficients rounded to float32)
        ln x = e * ln2 + (2 s) * p
    (the atanh series ln m = 2 atanh(s) = 2 (s + s^3/3 + ...), |s| <= 0.1716,
    truncated after s^9: the dropped terms are below 4e-10 relative)."""
    x = np.asarray(x, _F)
    bits = x.view(np.uint32)
    e = ((bits >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int32) - 127
    m = ((bits & np.uint32(0x007FFFFF)) | np.uint32(0x3F800000)).view(_F)
    big = m > _SQRT2
    m = np.where(big, m * _F(0.5), m).astype(_F)
    e = np.where(big, e + 1, e)
    s = ((m - _F(1.0)) / (m + _F(1.0))).astype(_F)
    t = (s * s).astype(_F)
    p = (t * _C[4]).astype(_F)
    p = ((p + _C[3]) * t).astype(_F)
    p = ((p + _C[2]) * t).astype(_F)
    p = ((p + _C[1]) * t).astype(_F)
    p = (p + _C[0]).astype(_F)
    return ((e.astype(_F) * _LN2).astype(_F) + ((s + s).astype(_F) * p).astype(_F)).astype(_F)


def gumbel_f32(seed: int, pos: int, vocab: int):
    """Gumbel noise G(seed, pos, v) for v < vocab, float32 [vocab]."""
    n4 = (vocab + 3) // 4
    ctr = np.zeros((n4, 4), np.uint64)
    ctr[:, 0] = np.arange(n4)
    ctr[:, 1] = np.uint64(pos & _MASK)
    key = np.array([seed & _MASK, (seed >> 32) & _MASK], np.uint64)
    words = philox4x32_10(ctr, key).reshape(-1)[:vocab]
    u = (((words >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(_F) * _F(2.0 ** -24)).astype(_F)
    return (-log_f32(-log_f32(u))).astype(_F)


def sampled_scores(logits_row, temperature: float, seed: int, pos: int):
    """float32 scores whose argmax is the draw (x * (1/T) + G); T <= 0: x."""
    x = np.asarray(logits_row, _F)
    t = _F(temperature)
    if not (np.isfinite(t) and t > 0):
        return x
    inv_t = _F(1.0) / t
    return ((x * inv_t).astype(_F) + gumbel_f32(seed, pos, x.shape[0])).astype(_F)


def sampled_draws(logits, vc, depth, temperature, seed):
    """logits [B*N][vocab]; vc [B]; depth [B][N]; temperature [B]; seed [B]
    (uint64). Returns the draws, int32 [B][N]."""
    depth = np.asarray(depth)
    B, N = depth.shape
    out = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(N):
            pos = int(vc[b]) + int(depth[b, i]) + 1
            sc = sampled_scores(logits[b * N + i], float(temperature[b]), int(seed[b]), pos)
            out[b, i] = _argmax.row_argmax(sc[None])[0]
    return out


def sampled_walk(parents, draft_tokens, logits, vc, depth, temperature, seed):
    """The draws, then the greedy walk over them. Returns (draws [B][N],
    accept_len [B], accepted_path [B][N], accepted_tokens [B][N])."""
    draws = sampled_draws(logits, vc, depth, temperature, seed)
    alen, path, tok = _walk.greedy_walk_batch(parents, draft_tokens, draws)
    return draws, alen, path, tok
