"""Pins of the top-k selection oracle (oracle/selection.py) against brute force and closed forms:
a Python sort of (-score, position) on small rows with many ties, signed zeros and infinities;
the order of the float keys; rows shorter than K; the length clamp."""
import math

import numpy as np
import pytest

from oracle.selection import order_keys, topk_select


def _brute(row, K, n):
    order = sorted(range(n), key=lambda j: (-float(row[j]), j))
    return order[:K] + [-1] * (K - min(K, n))


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_with_ties_zeros_and_infinities(seed):
    rng = np.random.default_rng(seed)
    T, S = 9, int(rng.integers(1, 70))
    pool = np.array([-np.inf, -3.5, -1.0, -0.0, 0.0, 0.25, 1.0, 1.0 + 2 ** -23, 7.0, np.inf], dtype=np.float32)
    scores = pool[rng.integers(0, len(pool), size=(T, S))]
    K = int(rng.integers(1, 2 * S + 2))
    lengths = rng.integers(-3, S + 5, size=T)
    got = topk_select(scores, K, lengths)
    for t in range(T):
        n = min(max(int(lengths[t]), 0), S)
        assert got[t].tolist() == _brute(scores[t], K, n), (t, n, K)


def test_order_keys_follow_the_float_order():
    vals = np.array([-np.inf, -3.4e38, -2.0, -1.0, -1e-30, -1e-45, 0.0, 1e-45, 1e-38, 0.5, 1.0, 3.4e38, np.inf],
                    dtype=np.float32)
    k = order_keys(vals)
    assert (np.diff(k) > 0).all()
    assert order_keys(np.array([-0.0], dtype=np.float32))[0] == order_keys(np.array([0.0], dtype=np.float32))[0]


def test_closed_forms():
    S, K = 50, 8
    scores = np.arange(S, dtype=np.float32)[None, :].repeat(3, axis=0)
    scores[1] = -scores[1]                      # descending row: best are the first positions
    scores[2] = 1.0                             # all equal: lowest positions first
    got = topk_select(scores, K)
    assert got[0].tolist() == list(range(S - 1, S - 1 - K, -1))
    assert got[1].tolist() == list(range(K))
    assert got[2].tolist() == list(range(K))


def test_short_rows_pad_with_minus_one_and_lengths_clamp():
    rng = np.random.default_rng(3)
    scores = rng.standard_normal((4, 30)).astype(np.float32)
    got = topk_select(scores, 40, lengths=[0, 5, 30, 99])
    assert (got[0] == -1).all()
    assert sorted(got[1, :5].tolist()) == list(range(5)) and (got[1, 5:] == -1).all()
    for t in (2, 3):   # a length past S clamps to S: every position, best first
        assert got[t, :30].tolist() == np.argsort(-scores[t], kind="stable").tolist()
        assert (got[t, 30:] == -1).all()
    vals = scores[3][got[3, :30]]
    assert (np.diff(vals) <= 0).all() and not math.isnan(float(vals.sum()))
