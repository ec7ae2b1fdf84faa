"""Pins for the SnapKV oracle: probability mass, a hand-worked two-token case,
a library routine (torch softmax with a causal mask), the pooling against
scipy's maximum filter, and the selection/compaction invariants."""
import math

import numpy as np
import pytest
import scipy.ndimage
import torch

from oracle.snapkv import compact, keep_positions, max_pool, window_scores


@pytest.mark.parametrize("seed", range(4))
def test_total_mass_is_rows_times_heads(seed):
    g = np.random.default_rng(seed)
    W, G, D, L = 5, 3, 8, 40
    A = window_scores(g.standard_normal((W, G, D)), g.standard_normal((L, D)), 0.35)
    assert abs(A.sum() - W * G) < 1e-12
    assert np.all(A >= 0)


def test_hand_worked_two_rows():
    # L = W = 2, one head, D = 1, scale 1.  Row 0 (position 0) sees only key 0,
    # so it puts mass 1 there.  Row 1 sees keys 0, 1 with logits q1*k0, q1*k1.
    q = np.array([[[0.7]], [[2.0]]])
    k = np.array([[0.5], [-1.0]])
    A = window_scores(q, k, 1.0)
    p0 = 1.0 / (1.0 + math.exp(-(2.0 * 0.5 - 2.0 * -1.0)))
    assert np.allclose(A, [1.0 + p0, 1.0 - p0], atol=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_matches_torch_causal_softmax(seed):
    g = np.random.default_rng(10 + seed)
    W, G, D, L = 6, 4, 16, 50
    q, k = g.standard_normal((W, G, D)), g.standard_normal((L, D))
    scale = 1 / math.sqrt(D)
    s = torch.einsum("wgd,ld->wgl", torch.from_numpy(q), torch.from_numpy(k)) * scale
    qpos = torch.arange(L - W, L)[:, None, None]
    s = s.masked_fill(torch.arange(L)[None, None, :] > qpos, float("-inf"))
    ref = torch.softmax(s, dim=-1).sum(dim=(0, 1)).numpy()
    assert np.allclose(window_scores(q, k, scale), ref, atol=1e-12)


@pytest.mark.parametrize("kernel", [1, 3, 7, 9])
def test_max_pool_matches_scipy_maximum_filter(kernel):
    a = np.random.default_rng(kernel).standard_normal(57)
    ref = scipy.ndimage.maximum_filter1d(a, size=kernel, mode="nearest")
    assert np.array_equal(max_pool(a, kernel), ref)


def test_max_pool_delta_and_identity():
    a = np.zeros(12)
    a[5] = 1.0
    assert np.nonzero(max_pool(a, 7))[0].tolist() == [2, 3, 4, 5, 6, 7, 8]
    a[0] = 2.0
    assert max_pool(a, 7)[:4].tolist() == [2.0, 2.0, 2.0, 2.0]
    b = np.random.default_rng(0).standard_normal(9)
    assert np.array_equal(max_pool(b, 1), b)


def test_keep_positions_rules():
    L, R = 30, 4
    A = np.arange(L, dtype=float)[::-1].copy()   # older is better
    kept = keep_positions(A, L, R, keep=5, kernel=1)
    assert kept.tolist() == [0, 1, 2, 3, 4, 26, 27, 28, 29]
    # everything kept when the budget covers the candidates
    assert keep_positions(A, L, R, keep=26, kernel=7).tolist() == list(range(L))
    assert keep_positions(A, L, R, keep=100, kernel=7).tolist() == list(range(L))
    # pooled plateaus: ties go to the lower position
    B = np.zeros(L)
    B[10] = 1.0
    kept = keep_positions(B, L, R, keep=3, kernel=7)
    assert kept.tolist() == [7, 8, 9, 26, 27, 28, 29]


@pytest.mark.parametrize("seed", range(3))
def test_compaction_preserves_rows_and_positions(seed):
    g = np.random.default_rng(seed)
    W, G, D, L, keep = 4, 2, 8, 64, 10
    q = g.standard_normal((W, G, D))
    kb = g.integers(0, 2 ** 16, size=(L, D), dtype=np.uint16)   # arbitrary bit patterns
    vb = g.integers(0, 2 ** 16, size=(L, D), dtype=np.uint16)
    kf = g.standard_normal((L, D))
    kept = keep_positions(window_scores(q, kf, 0.3), L, W, keep, kernel=7)
    ck, cv, pos = compact(kb, vb, kept)
    assert len(pos) == keep + W
    assert np.all(np.diff(pos) > 0)
    assert pos[-W:].tolist() == list(range(L - W, L))
    for i, p in enumerate(pos):
        assert ck[i].tobytes() == kb[p].tobytes() and cv[i].tobytes() == vb[p].tobytes()
