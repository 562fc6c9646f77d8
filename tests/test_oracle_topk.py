"""Pins of the oracle's top-k selection against an independent formulation
(a position is selected iff fewer than K valid positions beat it), hand-worked
cases and invariants.  CPU only."""
import math

import numpy as np
import pytest

from oracle import oracle as orc


def _beats(x, q, y, p):
    """score x at position q ranks above score y at position p (NaN lowest,
    -0 == +0, ties to the lower position)"""
    xn, yn = math.isnan(x), math.isnan(y)
    if xn != yn:
        return yn
    if not xn and x != y:
        return x > y
    return q < p


def _brute(scores, end_pos, K):
    B, S = scores.shape
    out = np.full((B, K), -1, np.int32)
    for b in range(B):
        T = min(max(int(end_pos[b]), 0), S)
        row = [float(v) for v in scores[b, :T]]
        sel = [p for p in range(T)
               if sum(1 for q in range(T) if q != p and _beats(row[q], q, row[p], p)) < K]
        out[b, :len(sel)] = sel
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    B, S = 3, 40
    scores = rng.standard_normal((B, S)).astype(np.float32)
    # ties, infinities, signed zeros and NaN
    scores[0, 5:12] = 0.5
    scores[1, ::7] = -0.0
    scores[1, 3::7] = 0.0
    scores[2, 4] = np.inf
    scores[2, 9] = -np.inf
    scores[2, 11] = np.nan
    scores[2, 30] = np.nan
    ends = np.array([40, 23, 37])
    for K in (1, 5, 12, 23, 40, 45):
        assert np.array_equal(orc.topk_select(scores, ends, K), _brute(scores, ends, K)), K


def test_topk_hand_worked():
    s = np.array([[1.0, 3.0, 3.0, -np.inf, np.nan, 2.0, -0.0, 0.0]], np.float32)
    # order: 3.0@1, 3.0@2, 2.0@5, 1.0@0, -0.0@6, 0.0@7 (equal: lower first), -inf@3, NaN@4
    assert orc.topk_select(s, [8], 3).tolist() == [[1, 2, 5]]
    assert orc.topk_select(s, [8], 5).tolist() == [[0, 1, 2, 5, 6]]
    assert orc.topk_select(s, [8], 7).tolist() == [[0, 1, 2, 3, 5, 6, 7]]
    assert orc.topk_select(s, [8], 8).tolist() == [[0, 1, 2, 3, 4, 5, 6, 7]]
    assert orc.topk_select(s, [4], 8).tolist() == [[0, 1, 2, 3, -1, -1, -1, -1]]
    assert orc.topk_select(s, [0], 2).tolist() == [[-1, -1]]


def test_topk_all_equal_takes_the_first_positions():
    s = np.full((2, 100), 7.25, np.float32)
    assert orc.topk_select(s, [100, 60], 10).tolist() == [list(range(10))] * 2


def test_topk_selected_outrank_the_rest():
    rng = np.random.default_rng(9)
    s = np.round(rng.standard_normal((4, 3000)) * 4).astype(np.float32)   # many ties
    ends = np.array([3000, 2999, 1500, 7])
    K = 500
    sel = orc.topk_select(s, ends, K)
    for b in range(4):
        T = int(ends[b])
        chosen = sel[b][sel[b] >= 0]
        assert chosen.size == min(K, T) and np.all(np.diff(chosen) > 0)
        rest = np.setdiff1d(np.arange(T), chosen)
        if rest.size:
            worst = min(chosen, key=lambda p: (s[b, p], -p))
            best = max(rest, key=lambda p: (s[b, p], -p))
            assert (s[b, worst], -worst) > (s[b, best], -best)
