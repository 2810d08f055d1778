"""Pins for oracle.sampling: the Philox4x32-10 known answers, the float32
logarithm against math.log, the uniform's exactness, the Gumbel-max draw's
distribution against softmax(x / T), and the page's keying rules (by position,
never by row; plain decoding's draw is the one accepted at each position)."""
import math

import numpy as np
import pytest
from scipy.stats import chisquare

from oracle import sampling as S
from oracle import walk as W
from tests.conftest import GOLDEN


def _kat():
    vals = {}
    with open(f"{GOLDEN}/philox4x32_10_kat.txt") as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":")
            vals[k.strip()] = [int(x, 16) for x in v.split()]
    return [(vals[f"ctr{i}"], vals[f"key{i}"], vals[f"out{i}"]) for i in range(3)]


@pytest.mark.parametrize("ctr, key, out", _kat())
def test_philox_known_answers(ctr, key, out):
    got = S.philox4x32_10(np.array(ctr, np.uint64), np.array(key, np.uint64))
    assert [int(x) for x in got] == out


def test_philox_is_vectorised_consistently():
    rng = np.random.default_rng(80)
    ctr = rng.integers(0, 2 ** 32, size=(50, 4), dtype=np.uint64)
    key = rng.integers(0, 2 ** 32, size=2, dtype=np.uint64)
    batch = S.philox4x32_10(ctr, key)
    one = np.stack([S.philox4x32_10(c, key) for c in ctr])
    assert (batch == one).all()


def test_log_f32_against_math_log():
    rng = np.random.default_rng(81)
    xs = np.concatenate([
        (np.arange(1, 2 ** 12, dtype=np.float64) * 2.0 ** -12),             # (0, 1)
        rng.uniform(2.0 ** -24, 1.0, 20000), rng.uniform(1.0, 20.0, 20000),
        np.array([2.0 ** -24, 2.0 ** -20, 0.5, 1.0, 2.0, math.sqrt(2.0), 16.6])]).astype(np.float32)
    got = S.log_f32(xs).astype(np.float64)
    ref = np.log(xs.astype(np.float64))
    err = np.abs(got - ref)
    # within a few float32 rounding steps of the result (absolute near x = 1)
    assert (err <= 4 * 2.0 ** -24 * np.maximum(np.abs(ref), 0.25)).all(), float(err.max())
    assert S.log_f32(np.float32(1.0)) == 0.0


def test_uniform_is_exact_and_open():
    words = S.philox4x32_10(np.stack([np.arange(4096), np.full(4096, 7), np.zeros(4096), np.zeros(4096)], 1),
                            np.array([123, 456])).reshape(-1)
    u = ((words >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(np.float32) * np.float32(2.0 ** -24)
    k = u.astype(np.float64) * 2 ** 24
    assert (k == np.round(k)).all() and (k.astype(np.int64) % 2 == 1).all()
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.01


@pytest.mark.parametrize("temperature", [1.0, 0.7, 2.5])
def test_draws_follow_softmax(temperature):
    """Gumbel-max: over many positions the draw of one row is distributed as
    softmax(x / T) (chi-square, fixed seeds)."""
    x = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4], np.float32)
    n = 30000
    counts = np.zeros(len(x))
    for pos in range(n):
        counts[int(np.argmax(S.sampled_scores(x, temperature, 99, pos)))] += 1
    p = np.exp(x.astype(np.float64) / temperature)
    p /= p.sum()
    assert chisquare(counts, n * p).pvalue > 1e-3


def test_zero_temperature_is_argmax():
    rng = np.random.default_rng(82)
    lg = rng.standard_normal((6, 300)).astype(np.float32)
    d = S.sampled_draws(lg, [10], np.arange(6)[None], [0.0], [5])
    assert d[0].tolist() == np.argmax(lg, axis=1).tolist()


def test_keyed_by_position_not_row():
    """Rows at the same depth (same predicted position) with the same logits
    draw the same token; moving rows around moves their draws with them."""
    rng = np.random.default_rng(83)
    vocab = 500
    lg = rng.standard_normal((1, vocab)).astype(np.float32)
    logits = np.repeat(lg, 6, axis=0)
    depth = np.array([[0, 1, 1, 2, 2, 2]])
    d = S.sampled_draws(logits, [40], depth, [1.0], [2024])[0]
    assert d[1] == d[2] and d[3] == d[4] == d[5]
    perm = [3, 0, 5, 1, 4, 2]
    d2 = S.sampled_draws(logits[perm], [40], depth[:, perm], [1.0], [2024])[0]
    assert d2.tolist() == d[perm].tolist()
    # positions matter: one row's draw over many positions is not constant
    assert len({int(np.argmax(S.sampled_scores(lg[0], 1.0, 2024, p))) for p in range(40)}) > 5


def test_chain_accepts_plain_decoding_draws():
    """The page: the token accepted at every position is the one plain decoding
    samples there. A chain whose drafts are plain decoding's draws (position
    vc + t + 1 for node t) is accepted whole, with those tokens."""
    rng = np.random.default_rng(84)
    N, vocab, vc, seed, T = 7, 64, 300, 77, 0.9
    logits = rng.standard_normal((N, vocab)).astype(np.float32)
    plain = [int(np.argmax(S.sampled_scores(logits[t], T, seed, vc + t + 1))) for t in range(N)]
    parents = np.array([list(range(-1, N - 1))])
    draft = np.array([[0] + plain[:-1]])               # node t drafts the token at position vc + t
    depth = np.arange(N)[None]
    draws, alen, path, tok = S.sampled_walk(parents, draft, logits, [vc], depth, [T], [seed])
    assert draws[0].tolist() == plain
    assert alen[0] == N and path[0].tolist() == list(range(N)) and tok[0].tolist() == plain
    ref = W.greedy_walk(parents[0], draft[0], draws[0])
    assert ref[0] == N
