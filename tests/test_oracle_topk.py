"""Pins for the oracle's top-k: brute force over all subsets, constructed ties."""
import itertools

import numpy as np
import pytest

from oracle.topk import rank_order, top_k


def brute_force_topk(scores, k):
    """The unique k-subset S with: every member beats every non-member, where
    i beats j iff s_i > s_j, or s_i == s_j and i < j.  Found by enumeration."""
    n = len(scores)
    found = []
    for S in itertools.combinations(range(n), k):
        inside = set(S)
        ok = all((scores[i] > scores[j]) or (scores[i] == scores[j] and i < j)
                 for i in inside for j in range(n) if j not in inside)
        if ok:
            found.append(S)
    assert len(found) == 1
    return np.array(found[0], dtype=np.int64)


@pytest.mark.parametrize("seed", range(20))
def test_topk_matches_brute_force_random(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 10))
    # few distinct values -> many ties and plateaus
    s = g.integers(-2, 3, size=n).astype(np.float64) * 0.5
    for k in range(0, n + 1):
        assert np.array_equal(top_k(s, k), brute_force_topk(list(s), k))


def test_topk_ties_go_to_lower_index():
    s = np.array([1.0, 3.0, 3.0, 3.0, 0.0])
    assert top_k(s, 2).tolist() == [1, 2]
    assert top_k(s, 3).tolist() == [1, 2, 3]
    assert top_k(s, 4).tolist() == [0, 1, 2, 3]


def test_topk_signed_zero_is_a_tie():
    s = np.array([-0.0, 0.0, -0.0])
    assert top_k(s, 1).tolist() == [0]
    assert top_k(s, 2).tolist() == [0, 1]


def test_rank_order_is_a_total_order_with_index_key():
    s = np.array([2.0, 5.0, 2.0, 5.0])
    idx = np.array([40, 30, 20, 10])
    # score 5 first (index 10 before 30), then score 2 (index 20 before 40)
    assert rank_order(s, idx).tolist() == [3, 1, 2, 0]


def test_topk_k_larger_than_n_returns_all():
    assert top_k(np.array([3.0, 1.0]), 5).tolist() == [0, 1]
