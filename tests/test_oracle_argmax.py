"""Pins for oracle.argmax: a pure-Python scan on small rows, the tie, NaN,
signed-zero and infinity cases, and the worked example's walk fed by logits."""
import math

import numpy as np
import pytest

from oracle import argmax as A
from oracle import walk as W


def _scan(row):
    """First index of the largest value, a NaN counting as larger than any
    number (the first NaN wins), written as a plain loop."""
    best_i, best = 0, row[0]
    for i, v in enumerate(row):
        if math.isnan(best):
            break
        if math.isnan(v) or v > best:
            best_i, best = i, v
    return best_i


def test_matches_plain_scan_with_many_ties():
    rng = np.random.default_rng(21)
    for _ in range(300):
        vocab = int(rng.integers(1, 40))
        rows = rng.integers(-3, 4, size=(int(rng.integers(1, 6)), vocab)).astype(np.float32)  # frequent ties
        got = A.row_argmax(rows)
        assert got.dtype == np.int32
        assert got.tolist() == [_scan([float(v) for v in r]) for r in rows]


def test_matches_plain_scan_on_normal_rows():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((50, 1000), dtype=np.float32)
    assert A.row_argmax(x).tolist() == [_scan([float(v) for v in r]) for r in x]


@pytest.mark.parametrize("row, expect", [
    ([5.0, 5.0, 5.0], 0),                        # all equal: the lowest index
    ([1.0, 7.0, 3.0, 7.0], 1),                   # tie: the lowest index
    ([-0.0, 0.0], 0),                            # -0 == +0
    ([0.0, -0.0], 0),
    ([-math.inf, -math.inf], 0),
    ([1.0, math.inf, math.inf], 1),
    ([2.0, math.nan, 9.0, math.nan], 1),         # the first NaN wins
    ([math.inf, math.nan], 1),                   # NaN above +inf
    ([-1.0], 0),
])
def test_special_cases(row, expect):
    assert A.row_argmax(np.array([row], np.float32)).tolist() == [expect]


def test_planted_maximum():
    """A row whose one entry exceeds every N(0,1) draw by far has that entry
    as its argmax (the synthetic logits plant the target this way)."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal((64, 5000), dtype=np.float32)
    t = rng.integers(0, 5000, 64)
    x[np.arange(64), t] = 20.0
    assert A.row_argmax(x).tolist() == t.tolist()


def test_worked_example_walk_from_logits(golden):
    """The (5, 4, 8) iteration: argmax over all 8 rows, then the walk; nodes
    0, 2, 5, 6 accept (accept_len 4)."""
    g = golden("accept_0_2_5_6.txt")
    n = len(g["parents"])
    vocab = 128
    rng = np.random.default_rng(24)
    logits = rng.standard_normal((n, vocab), dtype=np.float32)
    logits[np.arange(n), g["target_argmax"]] = 50.0
    arg, alen, path, tok = A.greedy_walk_from_logits(np.array([g["parents"]]), np.array([g["draft"]]), logits)
    assert arg[0].tolist() == g["target_argmax"]
    assert alen[0] == g["accept_len"][0]
    assert path[0].tolist() == g["accepted_path"]
    assert tok[0].tolist() == g["accepted_tokens"]
    ref = W.greedy_walk(g["parents"], g["draft"], g["target_argmax"])
    assert alen[0] == ref[0] and (path[0] == ref[1]).all()


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        A.row_argmax(np.zeros((3,), np.float32))
    with pytest.raises(ValueError):
        A.row_argmax(np.zeros((3, 0), np.float32))
