"""Pins for the attention oracle: a library routine (torch SDPA in float64),
closed forms, the split/merge identity, permutation invariance, and the
full-budget Quest view reducing to dense attention."""
import math

import numpy as np
import pytest
import torch

from oracle.attention import attend
from oracle.quest import page_minmax, quest_bound, quest_k_pages, quest_select, selected_tokens


@pytest.mark.parametrize("seed", range(6))
def test_matches_torch_sdpa_float64(seed):
    g = np.random.default_rng(seed)
    G, T, D = int(g.integers(1, 9)), int(g.integers(1, 70)), 16
    q, k, v = g.standard_normal((G, D)), g.standard_normal((T, D)), g.standard_normal((T, D))
    scale = 1 / math.sqrt(D)
    out, lse = attend(q, k, v, scale)
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, 0].numpy()
    assert np.allclose(out, ref, atol=1e-12, rtol=1e-12)
    ref_lse = torch.logsumexp(torch.from_numpy(scale * q @ k.T), dim=1).numpy()
    assert np.allclose(lse, ref_lse, atol=1e-12)


def test_constant_values_give_that_value():
    g = np.random.default_rng(1)
    q, k = g.standard_normal((3, 8)), g.standard_normal((50, 8))
    v = np.tile(np.arange(8.0), (50, 1))
    out, _ = attend(q, k, v, 0.3)
    assert np.allclose(out, np.arange(8.0)[None].repeat(3, 0), atol=1e-13)


def test_zero_query_is_uniform_average_and_log_count():
    g = np.random.default_rng(2)
    k, v = g.standard_normal((33, 4)), g.standard_normal((33, 4))
    out, lse = attend(np.zeros((1, 4)), k, v, 1.0)
    assert np.allclose(out[0], v.mean(axis=0), atol=1e-14)
    assert abs(lse[0] - math.log(33)) < 1e-14


def test_two_tokens_closed_form():
    q = np.array([[1.0, 0.0]])
    k = np.array([[2.0, 0.0], [-1.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0]])
    out, lse = attend(q, k, v, 0.5)          # logits 1.0 and -0.5
    w0 = 1.0 / (1.0 + math.exp(-1.5))
    assert np.allclose(out[0], [w0, 1 - w0], atol=1e-15)
    assert abs(lse[0] - math.log(math.exp(1.0) + math.exp(-0.5))) < 1e-15


@pytest.mark.parametrize("cut", [1, 7, 40, 63])
def test_split_and_lse_merge_identity(cut):
    g = np.random.default_rng(cut)
    q, k, v = g.standard_normal((4, 8)), g.standard_normal((64, 8)), g.standard_normal((64, 8))
    o, l = attend(q, k, v, 0.35)
    o1, l1 = attend(q, k[:cut], v[:cut], 0.35)
    o2, l2 = attend(q, k[cut:], v[cut:], 0.35)
    M = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - M), np.exp(l2 - M)
    merged = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None]
    assert np.allclose(merged, o, atol=1e-13)
    assert np.allclose(M + np.log(w1 + w2), l, atol=1e-13)


def test_permutation_invariance():
    g = np.random.default_rng(3)
    q, k, v = g.standard_normal((2, 8)), g.standard_normal((29, 8)), g.standard_normal((29, 8))
    perm = g.permutation(29)
    a, la = attend(q, k, v, 0.4)
    b, lb = attend(q, k[perm], v[perm], 0.4)
    assert np.allclose(a, b, atol=1e-13) and np.allclose(la, lb, atol=1e-13)


def test_empty_set():
    out, lse = attend(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_full_budget_quest_equals_dense_attention():
    g = np.random.default_rng(4)
    G, D, T = 4, 16, 16 * 12 + 3
    q, k, v = g.standard_normal((G, D)), g.standard_normal((T, D)), g.standard_normal((T, D))
    kmin, kmax = page_minmax(k)
    sel = quest_select(quest_bound(q, kmin, kmax), quest_k_pages(10 ** 9))
    tok = selected_tokens(sel, T)
    assert tok.tolist() == list(range(T))
    out, lse = attend(q, k[tok], v[tok], 0.25)
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.25)[0, 0].numpy()
    assert np.allclose(out, ref, atol=1e-12)
