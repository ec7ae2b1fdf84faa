"""Pins of the cross-layer selection-reuse oracle (oracle/omnikv.py) against
closed forms, library routines and a hand-built case where reuse and a
layer's own selection differ."""
import math

import numpy as np
import pytest

from oracle.omnikv import filter_pages, omnikv_layers, source_layer
from oracle.quest import quest_bound, page_minmax, quest_k_pages, quest_select

torch = pytest.importorskip("torch")


def _sdpa(q, k, v, scale):
    """torch softmax attention in float64 (library routine)."""
    qt = torch.tensor(np.asarray(q), dtype=torch.float64)[None, :, None, :]
    kt = torch.tensor(np.asarray(k), dtype=torch.float64)[None, None].expand(1, qt.shape[1], -1, -1)
    vt = torch.tensor(np.asarray(v), dtype=torch.float64)[None, None].expand(1, qt.shape[1], -1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return out[0, :, 0].numpy()


def _layers(seed, L, T=200, G=4, D=16):
    rng = np.random.default_rng(seed)
    qs = [rng.standard_normal((G, D)) for _ in range(L)]
    ks = [rng.standard_normal((T, D)) for _ in range(L)]
    vs = [rng.standard_normal((T, D)) for _ in range(L)]
    return qs, ks, vs


def test_source_layer_is_the_latest_filter_at_or_before():
    assert [source_layer(x, (0, 2)) for x in range(4)] == [0, 0, 2, 2]
    assert [source_layer(x, (0,)) for x in range(3)] == [0, 0, 0]
    with pytest.raises(ValueError):
        source_layer(0, (1,))


@pytest.mark.parametrize("seed", range(3))
def test_full_budget_is_dense_attention_per_layer(seed):
    qs, ks, vs = _layers(seed, 3)
    scale = 1 / math.sqrt(16)
    res = omnikv_layers(qs, ks, vs, (0,), 10 ** 9, scale)
    for layer, (pages, out, _) in enumerate(res):
        assert np.array_equal(pages, np.arange(13))           # ceil(200 / 16) pages
        assert np.allclose(out, _sdpa(qs[layer], ks[layer], vs[layer], scale), atol=1e-12)


def test_identical_layers_reproduce_the_filter_layer():
    qs, ks, vs = _layers(7, 1)
    res = omnikv_layers(qs * 4, ks * 4, vs * 4, (0,), 48, 0.25)
    for pages, out, lse in res[1:]:
        assert np.array_equal(pages, res[0][0])
        assert np.array_equal(out, res[0][1]) and np.array_equal(lse, res[0][2])


def test_reuse_takes_the_filter_layers_pages_not_the_layers_own():
    """Three pages of 16 tokens, a budget of two pages (the last page is
    forced, one more is chosen).  Layer 0's keys make page 0 the best for its
    query; layer 1's keys would make page 1 its own choice.  Layer 1 must
    attend over its own tokens of pages {0, 2}."""
    D, T = 4, 48
    q = np.array([[1.0, 0.0, 0.0, 0.0]])
    k0 = np.zeros((T, D))
    k0[0:16, 0] = 5.0                  # page 0 wins for layer 0
    k1 = np.zeros((T, D))
    k1[16:32, 0] = 5.0                 # page 1 would win for layer 1
    rng = np.random.default_rng(0)
    v0, v1 = rng.standard_normal((T, D)), rng.standard_normal((T, D))
    res = omnikv_layers([q, q], [k0, k1], [v0, v1], (0,), 32, 0.5)
    assert list(res[0][0]) == [0, 2] and list(res[1][0]) == [0, 2]
    tok = np.r_[0:16, 32:48]
    assert np.allclose(res[1][1], _sdpa(q, k1[tok], v1[tok], 0.5), atol=1e-12)
    other = np.r_[16:32, 32:48]
    assert not np.allclose(res[1][1], _sdpa(q, k1[other], v1[other], 0.5), atol=1e-6)
    # with layer 1 a filter layer too, it takes its own choice
    res2 = omnikv_layers([q, q], [k0, k1], [v0, v1], (0, 1), 32, 0.5)
    assert list(res2[1][0]) == [1, 2]


def test_every_layer_a_filter_is_per_layer_quest():
    qs, ks, vs = _layers(3, 3)
    res = omnikv_layers(qs, ks, vs, (0, 1, 2), 64, 0.25)
    for layer, (pages, _, _) in enumerate(res):
        U = quest_bound(qs[layer], *page_minmax(ks[layer]))
        assert np.array_equal(pages, quest_select(U, quest_k_pages(64)))


def test_filter_pages_is_the_quest_selection_of_that_layer():
    qs, ks, _ = _layers(5, 1)
    assert np.array_equal(filter_pages(qs[0], ks[0], 96),
                          quest_select(quest_bound(qs[0], *page_minmax(ks[0])), 6))
