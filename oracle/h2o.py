"""H2O heavy-hitter + recent-window eviction (oracle).

H2O keeps a running, accumulated attention score per retained token; every
decode step adds that step's attention to the scores and then decides which
token to delete, and the deletion is physical ("tokendh.com article",
sections "历史太长,会撑爆什么" and "把边界划在'生命周期'上").

Definitions used here (one sequence, one KV head with G query heads):

* a step appends the new token with score 0, attends over every retained
  token (the new one included) with softmax probabilities
  p[g,t] = exp(s[g,t] - lse[g]), and adds sum_g p[g,t] to score[t];
* if more than ``budget`` tokens are now held, one is evicted: the recent
  window (the ``recent`` largest logical positions, which include the new
  token) is protected; among the other tokens the one ranked last under
  (score desc, position asc) is evicted -- i.e. the lowest score, and among
  equal lowest scores the higher position;
* initial state (a reading: the pages do not say how the prefill scores
  arise): the column scores of the last ``window`` prefill query rows (the
  SnapKV window score without pooling) seed the scores; the ``recent`` newest
  positions plus the best ``budget - recent`` older ones by that score
  (position asc on ties) are kept.
"""
import dataclasses

import numpy as np

from .attention import attend, logits
from .snapkv import keep_positions, window_scores
from .topk import rank_order


@dataclasses.dataclass
class H2OState:
    pos: np.ndarray     # [n] logical positions (any order)
    k: np.ndarray       # [n][D] float64
    v: np.ndarray       # [n][D] float64
    score: np.ndarray   # [n] float64


def h2o_init(q_win, k, v, budget: int, recent: int, scale: float) -> H2OState:
    """State after prefill of L = len(k) tokens; q_win [W][G][D]."""
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L = k.shape[0]
    A = window_scores(q_win, k, scale)
    keep = keep_positions(A, L, recent, budget - recent, kernel=1)
    return H2OState(pos=keep.copy(), k=k[keep], v=v[keep], score=A[keep].copy())


def h2o_step(st: H2OState, q_group, k_new, v_new, new_pos: int,
             budget: int, recent: int, scale: float):
    """One decode step.  Returns (new_state, out [G][D], lse [G], evicted_pos),
    evicted_pos = -1 when nothing is evicted."""
    pos = np.concatenate([st.pos, [new_pos]]).astype(np.int64)
    k = np.vstack([st.k, np.asarray(k_new, dtype=np.float64)[None]])
    v = np.vstack([st.v, np.asarray(v_new, dtype=np.float64)[None]])
    score = np.concatenate([st.score, [0.0]])

    out, lse = attend(q_group, k, v, scale)
    p = np.exp(logits(q_group, k, scale) - lse[:, None])
    score = score + p.sum(axis=0)

    evicted = -1
    if len(pos) > budget:
        newest = np.argsort(pos)[::-1][:recent]          # the `recent` largest positions
        cand = np.setdiff1d(np.arange(len(pos)), newest)
        order = rank_order(score[cand], index=pos[cand])
        victim = cand[order[-1]]
        evicted = int(pos[victim])
        keep = np.ones(len(pos), dtype=bool)
        keep[victim] = False
        pos, k, v, score = pos[keep], k[keep], v[keep], score[keep]
    return H2OState(pos=pos, k=k, v=v, score=score), out, lse, evicted
