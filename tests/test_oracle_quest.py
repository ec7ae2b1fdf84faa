"""Pins for the Quest oracle: the bound property, the page-size-1 reduction to
exact top-k of the logits, a hand-worked bound, and the selection rules."""
import numpy as np
import pytest

from oracle.quest import page_minmax, quest_bound, quest_k_pages, quest_select, selected_tokens
from tests.test_oracle_topk import brute_force_topk


def test_hand_worked_bound():
    # Two query heads, D = 2; one page with keys (-1, 3) and (2, 0):
    #   kmin = (-1, 0), kmax = (2, 3)
    #   head 0, q = (1, -2):   d0: max(-1, 2) = 2      d1: max(-0, -6) = 0   -> 2
    #   head 1, q = (-1, 0.5): d0: max(1, -2) = 1      d1: max(0, 1.5) = 1.5 -> 2.5
    #   U = 4.5, while the best group-summed logit is max(-7 + 2.5, 2 - 2) = 0.
    q = np.array([[1.0, -2.0], [-1.0, 0.5]])
    keys = np.array([[-1.0, 3.0], [2.0, 0.0]])
    kmin, kmax = page_minmax(keys, page_size=2)
    assert kmin.tolist() == [[-1.0, 0.0]] and kmax.tolist() == [[2.0, 3.0]]
    assert quest_bound(q, kmin, kmax).tolist() == [4.5]


@pytest.mark.parametrize("seed", range(5))
def test_bound_dominates_every_key_of_its_page(seed):
    g = np.random.default_rng(seed)
    G, D, T, P = 4, 16, 16 * 9 + 5, 16       # ragged last page
    q = g.standard_normal((G, D))
    k = g.standard_normal((T, D))
    kmin, kmax = page_minmax(k, P)
    U = quest_bound(q, kmin, kmax)
    for p in range(len(U)):
        blk = k[p * P:(p + 1) * P]
        group_logit = (q @ blk.T).sum(axis=0)
        assert U[p] >= group_logit.max() - 1e-12
        for gi in range(G):   # per head as well
            Ug = quest_bound(q[gi:gi + 1], kmin[p:p + 1], kmax[p:p + 1])[0]
            assert Ug >= (q[gi] @ blk.T).max() - 1e-12


def test_page_minmax_are_attained_extremes_over_valid_tokens():
    g = np.random.default_rng(7)
    k = g.standard_normal((37, 8))           # pages of 16, 16, 5
    kmin, kmax = page_minmax(k, 16)
    assert kmin.shape == (3, 8)
    for p, (a, b) in enumerate([(0, 16), (16, 32), (32, 37)]):
        blk = k[a:b]
        assert np.all(blk >= kmin[p]) and np.all(blk <= kmax[p])
        for d in range(8):
            assert kmin[p, d] in blk[:, d] and kmax[p, d] in blk[:, d]


@pytest.mark.parametrize("seed", range(8))
def test_page_size_one_is_exact_topk_of_group_logits(seed):
    # With one token per page kmin = kmax = k, so the bound is the exact
    # group-summed logit and Quest becomes exact token top-k (newest forced).
    g = np.random.default_rng(seed)
    G, D, T = 2, 4, 9
    q = g.integers(-2, 3, size=(G, D)).astype(float)
    k = g.integers(-2, 3, size=(T, D)).astype(float)
    kmin, kmax = page_minmax(k, 1)
    U = quest_bound(q, kmin, kmax)
    exact = (q @ k.T).sum(axis=0)
    assert np.array_equal(U, exact)
    for kk in range(1, T + 1):
        sel = quest_select(U, kk)
        want = np.concatenate([brute_force_topk(list(exact[:T - 1]), kk - 1), [T - 1]]) \
            if kk < T else np.arange(T)
        assert np.array_equal(sel, want)


def test_selection_rules():
    U = np.array([5.0, 1.0, 7.0, 7.0, 2.0, -100.0])
    assert quest_select(U, 1).tolist() == [5]              # only the forced last page
    assert quest_select(U, 3).tolist() == [2, 3, 5]        # tie at 7: both; last forced
    assert quest_select(U, 4).tolist() == [0, 2, 3, 5]
    assert quest_select(U, 6).tolist() == [0, 1, 2, 3, 4, 5]
    assert quest_select(U, 99).tolist() == [0, 1, 2, 3, 4, 5]


def test_budget_to_pages():
    # A budget of 128 tokens at page size 16 is the "top-8 pages incl. last page" case.
    assert quest_k_pages(128) == 8
    assert quest_k_pages(2048) == 128
    assert quest_k_pages(4096) == 256
    assert quest_k_pages(15) == 1 and quest_k_pages(0) == 1


def test_selected_tokens_partial_last_page():
    assert selected_tokens([0, 2], ctx=37, page_size=16).tolist() == \
        list(range(0, 16)) + list(range(32, 37))


# ---- the max-aggregation variant --------------------------------------------

from oracle.quest import quest_bound_max  # noqa: E402


def test_max_bound_hand_worked():
    """Two query heads, one page of two keys, D = 2:
    head 0 (1, -1): per channel max(1*kmin, 1*kmax) + max(-kmin, -kmax)
    head 1 (-2, 0.5)."""
    k = np.array([[1.0, 2.0], [3.0, -1.0]])
    kmin, kmax = k.min(axis=0)[None], k.max(axis=0)[None]     # (1, -1), (3, 2)
    q = np.array([[1.0, -1.0], [-2.0, 0.5]])
    # head 0: 3 + 1 = 4;  head 1: max(-2, -6) + max(-0.5, 1) = -2 + 1 = -1
    assert np.allclose(quest_bound_max(q, kmin, kmax), [4.0])
    assert np.allclose(quest_bound(q, kmin, kmax), [3.0])


@pytest.mark.parametrize("seed", range(3))
def test_max_bound_dominates_every_heads_logit(seed):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((200, 32))
    q = rng.standard_normal((8, 32))
    U = quest_bound_max(q, *page_minmax(K))
    logits = q @ K.T                                          # [G][T]
    for p in range(len(U)):
        assert U[p] >= logits[:, p * 16:(p + 1) * 16].max() - 1e-9


def test_max_bound_page_size_one_is_the_exact_max_logit():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((40, 8))
    q = rng.standard_normal((4, 8))
    kmin, kmax = page_minmax(K, page_size=1)
    want = np.array([max(float(q[g] @ K[t]) for g in range(4)) for t in range(40)])
    assert np.allclose(quest_bound_max(q, kmin, kmax), want)


def test_max_bound_single_head_is_the_sum_bound():
    rng = np.random.default_rng(5)
    K = rng.standard_normal((100, 16))
    q = rng.standard_normal((1, 16))
    mm = page_minmax(K)
    assert np.array_equal(quest_bound_max(q, *mm), quest_bound(q, *mm))
