"""Pins of the span-pruning and sink + recent oracles (oracle/prune.py)."""
import numpy as np
import pytest

from oracle.prune import sink_recent_pages, span_keep_positions
from oracle.snapkv import keep_positions
from oracle.topk import top_k


def test_span_over_the_whole_prefix_is_snapkv_selection():
    """A span [0, L - W) keeping `keep` tokens is SnapKV's rule with window W."""
    rng = np.random.default_rng(0)
    A = rng.random(300)
    for kernel in (1, 3, 7):
        assert np.array_equal(span_keep_positions(A, 300, 0, 268, 100, kernel),
                              keep_positions(A, 300, 32, 100, kernel))


def test_keep_everything_or_nothing():
    A = np.random.default_rng(1).random(100)
    assert np.array_equal(span_keep_positions(A, 100, 20, 60, 40, 5), np.arange(100))
    assert np.array_equal(span_keep_positions(A, 100, 20, 60, 0, 5),
                          np.r_[0:20, 60:100])


def test_hand_worked_spike():
    """One spike at 30 in the span [20, 40), pool 3, keep 3: the spike and its
    two neighbours survive (ties of the plateau go to the lower position, so
    the next-best token, 10 away, loses to the plateau)."""
    A = np.zeros(50)
    A[30] = 5.0
    A[35] = 1.0
    got = span_keep_positions(A, 50, 20, 40, 3, 3)
    assert np.array_equal(got, np.r_[0:20, 29, 30, 31, 40:50])


def test_outside_positions_untouched_and_ascending():
    rng = np.random.default_rng(2)
    for _ in range(20):
        L = int(rng.integers(1, 400))
        s0, s1 = sorted(int(x) for x in rng.integers(-10, L + 10, size=2))
        keep = int(rng.integers(0, 50))
        k = int(rng.choice([1, 3, 7]))
        got = span_keep_positions(rng.random(L), L, s0, s1, keep, k)
        assert np.all(np.diff(got) > 0)
        lo, hi = max(0, min(s0, L)), max(max(0, min(s0, L)), min(s1, L))
        assert set(range(lo)) <= set(got) and set(range(hi, L)) <= set(got)
        assert len(got) == lo + min(keep, hi - lo) + (L - hi)


def test_span_selection_matches_brute_force_on_small_cases():
    rng = np.random.default_rng(3)
    for _ in range(30):
        L = int(rng.integers(5, 40))
        s0 = int(rng.integers(0, L))
        s1 = int(rng.integers(s0, L + 1))
        keep = int(rng.integers(0, s1 - s0 + 1))
        A = rng.integers(0, 4, size=L).astype(float)          # plenty of ties
        pooled = [max(A[max(s0, j - 1):min(s1, j + 2)]) for j in range(s0, s1)]
        order = sorted(range(s1 - s0), key=lambda i: (-pooled[i], i))[:keep]
        want = np.r_[0:s0, np.sort(np.asarray(order, dtype=int)) + s0, s1:L]
        assert np.array_equal(span_keep_positions(A, L, s0, s1, keep, 3), want)


@pytest.mark.parametrize("L,sink,recent,want", [
    (160, 1, 2, [0, 8, 9]),
    (161, 1, 2, [0, 9, 10]),
    (40, 2, 2, [0, 1, 2]),           # overlap: every page once
    (16, 1, 1, [0]),
    (0, 1, 1, []),
    (100, 0, 1, [6]),
])
def test_sink_recent_pages(L, sink, recent, want):
    assert list(sink_recent_pages(L, sink, recent)) == want
