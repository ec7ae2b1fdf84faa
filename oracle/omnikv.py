"""Cross-layer selection reuse, OmniKV-style (oracle).

Some layers decide which part of the history matters and hand that decision to
the later layers, which reuse it without deciding again ("tokendh.com article",
section "把边界划在'生命周期'上": OmniKV judges importance in certain layers and
passes the result to the following layers to reuse directly).

Definitions used here (one sequence, one KV head; L layers, each with its own
keys, values and query heads; a sorted set F of filter layers containing 0):

* the decision of filter layer f is its Quest page selection (``quest.py``:
  the group-summed page bound over f's own keys and queries, the top k-1
  pages plus the forced last page);
* layer l attends with its own queries over its own keys and values of the
  pages chosen by the latest filter layer f <= l (a reading: the pages say the
  decision is reused by the later layers, not how far; each filter layer
  starts a new decision);
* every layer sees the same positions (the layers of one model hold one
  token sequence), so a page means the same positions in every layer.
"""
import numpy as np

from .attention import attend
from .quest import page_minmax, quest_bound, quest_k_pages, quest_select, selected_tokens


def source_layer(layer: int, filters) -> int:
    """The filter layer whose decision layer ``layer`` reuses: the latest
    filter layer at or before it."""
    f = [x for x in sorted(filters) if x <= layer]
    if not f:
        raise ValueError("layer 0 must be a filter layer")
    return f[-1]


def filter_pages(q_group, k, budget_tokens: int) -> np.ndarray:
    """A filter layer's decision: its Quest page selection over its own keys
    k [T][D] with its query heads q_group [G][D]."""
    kmin, kmax = page_minmax(k)
    return quest_select(quest_bound(q_group, kmin, kmax), quest_k_pages(budget_tokens))


def omnikv_layers(qs, ks, vs, filters, budget_tokens: int, scale: float):
    """One decode step of one (sequence, KV head) through L layers.

    qs[l] [G][D], ks[l] / vs[l] [T][D] (every layer holds T tokens).
    Returns a list over layers of (pages used, out [G][D], lse [G])."""
    L = len(qs)
    T = np.asarray(ks[0]).shape[0]
    decided = {}
    res = []
    for layer in range(L):
        f = source_layer(layer, filters)
        if f not in decided:
            decided[f] = filter_pages(qs[f], ks[f], budget_tokens)
        pages = decided[f]
        tok = selected_tokens(pages, T)
        out, lse = attend(qs[layer], np.asarray(ks[layer])[tok], np.asarray(vs[layer])[tok], scale)
        res.append((pages, out, lse))
    return res
