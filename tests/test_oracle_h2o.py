"""Pins for the H2O oracle: a hand-worked step, mass conservation, the
no-eviction closed form (scores = summed step probabilities from torch's
softmax), and the protection/argmin rules checked by brute force."""
import numpy as np
import pytest
import torch

from oracle.h2o import H2OState, h2o_init, h2o_step
from oracle.snapkv import window_scores


def _state(pos, score, D=1, g=None):
    n = len(pos)
    k = np.zeros((n, D)) if g is None else g.standard_normal((n, D))
    v = np.arange(n * D, dtype=float).reshape(n, D) if g is None else g.standard_normal((n, D))
    return H2OState(pos=np.array(pos), k=k, v=v, score=np.array(score, dtype=float))


def test_hand_worked_step():
    # Two tokens held (positions 0 and 1, scores 0.5 and 0.2, all keys 0), budget 2,
    # recent window 1.  The new token (position 2, key 0) makes all logits 0:
    # each token gets 1/3.  Scores: 0.8333, 0.5333, 0.3333; position 2 is protected;
    # position 1 has the lowest candidate score and is evicted.
    st = _state([0, 1], [0.5, 0.2])
    st.v = np.array([[1.0], [2.0]])
    new, out, lse, ev = h2o_step(st, np.array([[1.0]]), np.array([0.0]), np.array([6.0]),
                                 new_pos=2, budget=2, recent=1, scale=1.0)
    assert ev == 1
    assert sorted(new.pos.tolist()) == [0, 2]
    got = dict(zip(new.pos.tolist(), new.score.tolist()))
    assert abs(got[0] - (0.5 + 1 / 3)) < 1e-15 and abs(got[2] - 1 / 3) < 1e-15
    assert abs(out[0, 0] - 3.0) < 1e-14
    assert abs(lse[0] - np.log(3.0)) < 1e-15


def test_equal_lowest_scores_evict_the_higher_position():
    st = _state([0, 1, 2], [0.0, 0.0, 0.0])
    new, _, _, ev = h2o_step(st, np.array([[0.0]]), np.array([0.0]), np.array([0.0]),
                             new_pos=3, budget=3, recent=1, scale=1.0)
    # all four receive 1/4; positions 0, 1, 2 tie as candidates -> evict 2
    assert ev == 2


@pytest.mark.parametrize("seed", range(5))
def test_mass_conservation_and_rules(seed):
    g = np.random.default_rng(seed)
    G, D, n, budget, recent = 4, 8, 20, 20, 5
    st = _state(list(g.permutation(40)[:n]), g.random(n), D=D, g=g)
    for step in range(6):
        new_pos = 100 + step
        q, kn, vn = g.standard_normal((G, D)), g.standard_normal(D), g.standard_normal(D)
        allpos = np.concatenate([st.pos, [new_pos]])
        K = torch.from_numpy(np.vstack([st.k, kn[None]]))
        # the step's probabilities from torch's softmax (summed over the group)
        p = torch.softmax(0.3 * torch.from_numpy(q) @ K.T, dim=-1).sum(dim=0).numpy()
        updated = np.concatenate([st.score, [0.0]]) + p
        new, out, lse, ev = h2o_step(st, q, kn, vn, new_pos, budget, recent, 0.3)
        assert ev != -1 and len(new.pos) == budget
        victim = int(np.nonzero(allpos == ev)[0][0])
        # mass conservation: sum after = sum before + G - victim's updated score
        assert abs(new.score.sum() - (st.score.sum() + G - updated[victim])) < 1e-12
        # protected window never evicted; victim is the brute-force argmin
        # (ties -> higher position) over the unprotected tokens
        newest = set(sorted(allpos.tolist())[-recent:])
        cands = [i for i in range(len(allpos)) if allpos[i] not in newest]
        best = min(cands, key=lambda i: (updated[i], -allpos[i]))
        assert victim == best
        st = new


def test_no_eviction_scores_are_summed_step_probabilities():
    g = np.random.default_rng(9)
    G, D, n0, steps = 2, 8, 6, 5
    st = _state(list(range(n0)), np.zeros(n0), D=D, g=g)
    keys, acc = [k for k in st.k], np.zeros(n0 + steps)
    for s in range(steps):
        q, kn, vn = g.standard_normal((G, D)), g.standard_normal(D), g.standard_normal(D)
        keys.append(kn)
        st, _, _, ev = h2o_step(st, q, kn, vn, n0 + s, budget=1000, recent=2, scale=0.4)
        assert ev == -1
        K = torch.from_numpy(np.array(keys))
        p = torch.softmax(0.4 * torch.from_numpy(q) @ K.T, dim=-1).sum(dim=0).numpy()
        acc[:len(p)] += p
    order = np.argsort(st.pos)
    assert np.allclose(st.score[order], acc, atol=1e-12)


def test_init_keeps_recent_and_heavy_hitters():
    g = np.random.default_rng(11)
    W, G, D, L, budget, recent = 4, 2, 8, 80, 24, 8
    q, k, v = g.standard_normal((W, G, D)), g.standard_normal((L, D)), g.standard_normal((L, D))
    st = h2o_init(q, k, v, budget, recent, 0.3)
    A = window_scores(q, k, 0.3)
    assert len(st.pos) == budget
    assert st.pos[-recent:].tolist() == list(range(L - recent, L))
    older = st.pos[:-recent]
    dropped = np.setdiff1d(np.arange(L - recent), older)
    assert A[older].min() >= A[dropped].max()
    assert np.array_equal(st.score, A[st.pos])
