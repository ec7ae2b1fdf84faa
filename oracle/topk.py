"""Exact top-k under one total order: score descending, then index ascending.

This is the tie rule for every selection of the path (Quest pages, SnapKV
positions, H2O eviction): among equal scores the lower index ranks first.
-0.0 and +0.0 compare equal (numeric comparison).  NaN is outside the contract.
"""
import numpy as np


def rank_order(scores, index=None) -> np.ndarray:
    """Positions into ``scores`` ordered by (score desc, index asc).
    ``index`` defaults to 0..n-1 and only breaks ties."""
    s = np.asarray(scores, dtype=np.float64)
    idx = np.arange(len(s)) if index is None else np.asarray(index)
    # np.lexsort sorts by the last key first; both keys ascending.
    return np.lexsort((idx, -s))


def top_k(scores, k, index=None) -> np.ndarray:
    """The k best positions under (score desc, index asc), returned in
    ascending position order.  k >= n returns all positions."""
    s = np.asarray(scores, dtype=np.float64)
    k = max(0, min(int(k), len(s)))
    return np.sort(rank_order(s, index)[:k])
