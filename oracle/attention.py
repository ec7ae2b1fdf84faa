"""Decode-step attention over a selected token set (oracle).

The attention of one decode query reads only the positions that the method's
view exposes ("SparseEngine：稀疏优先推理引擎", section "方法 / 关键模块":
AttentionView exposes the selected positions in one format; "tokendh.com
article", section "把边界划在'生命周期'上").  Over those tokens it is plain
softmax attention:

    s[g,t] = scale * q[g] . k[t]
    out[g] = sum_t softmax_t(s[g,:]) v[t]
    lse[g] = log sum_t exp(s[g,t])

computed two-pass (max, then normalised sum) in float64.  An empty token set
gives out = 0 and lse = -inf.
"""
import numpy as np


def logits(q_group, k_sel, scale: float):
    """s[g,t] = scale * q[g].k[t]  (float64)."""
    q = np.asarray(q_group, dtype=np.float64)
    k = np.asarray(k_sel, dtype=np.float64)
    return scale * (q @ k.T)


def attend(q_group, k_sel, v_sel, scale: float):
    """Softmax attention of queries [G][D] over keys/values [T][D].
    Returns (out [G][Dv], lse [G])."""
    q = np.asarray(q_group, dtype=np.float64)
    v = np.asarray(v_sel, dtype=np.float64)
    G = q.shape[0]
    if len(v) == 0:
        return np.zeros((G, v.shape[1] if v.ndim == 2 else q.shape[1])), np.full(G, -np.inf)
    s = logits(q, k_sel, scale)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ v) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse
