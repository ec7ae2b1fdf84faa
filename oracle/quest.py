"""Quest query-aware page selection (oracle).

Quest keeps the whole history and a small per-page summary, then picks, for
each query, the pages whose keys can score highest ("tokendh.com article",
section "历史太长,会撑爆什么": dynamic-sparse methods keep the full history
plus a summary index; Quest selects pages by the query).  KV is stored in
fixed-size pages of 16 tokens ("长程 agent 把显存撑爆以后", section
"四、为什么进不了 vLLM 一类的引擎").

Definitions used here:

* page summary: per page and channel d, kmin_d / kmax_d over the page's valid
  tokens (a partial last page uses only its valid tokens);
* upper bound of a page for one query head: sum_d max(q_d*kmin_d, q_d*kmax_d),
  which is >= q.k for every key of the page;
* GQA reading: the KV head's page score is the SUM of its query heads' bounds
  (an upper bound of the group-summed logit; all query heads of a KV head
  share one page selection); the alternative reading, the MAX of the query
  heads' bounds (an upper bound of every head's own logit), is
  ``quest_bound_max``, selectable as a flag;
* budget: k = max(1, floor(budget / 16)) pages per KV head; the last page
  (holding the newest token) is always selected and counts against k; the
  other k-1 are the best remaining pages under (score desc, page asc); if the
  sequence has <= k pages, all are selected; the result is in ascending order;
* the bound carries no 1/sqrt(D) factor (a positive scale does not change the
  ranking).
"""
import numpy as np

from .topk import top_k

PAGE = 16


def page_minmax(k_tokens, page_size: int = PAGE):
    """kmin, kmax [n_pages][D] of keys [T][D] (float64), over valid tokens."""
    k = np.asarray(k_tokens, dtype=np.float64)
    T, D = k.shape
    n_pages = -(-T // page_size)
    kmin = np.empty((n_pages, D))
    kmax = np.empty((n_pages, D))
    for p in range(n_pages):
        blk = k[p * page_size:min(T, (p + 1) * page_size)]
        kmin[p] = blk.min(axis=0)
        kmax[p] = blk.max(axis=0)
    return kmin, kmax


def quest_bound(q_group, kmin, kmax):
    """U[p] = sum over the group's query heads g and channels d of
    max(q[g,d]*kmin[p,d], q[g,d]*kmax[p,d]).  q_group [G][D]."""
    q = np.asarray(q_group, dtype=np.float64)
    lo = q[:, None, :] * np.asarray(kmin, dtype=np.float64)[None, :, :]   # [G][P][D]
    hi = q[:, None, :] * np.asarray(kmax, dtype=np.float64)[None, :, :]
    return np.maximum(lo, hi).sum(axis=(0, 2))


def quest_bound_max(q_group, kmin, kmax):
    """The max-aggregation variant of the bound (the alternative reading of
    how a KV head's query heads combine): U[p] = max over the group's query
    heads g of sum_d max(q[g,d]*kmin[p,d], q[g,d]*kmax[p,d]) -- each head's own
    upper bound, the largest of them.  q_group [G][D]."""
    q = np.asarray(q_group, dtype=np.float64)
    lo = q[:, None, :] * np.asarray(kmin, dtype=np.float64)[None, :, :]   # [G][P][D]
    hi = q[:, None, :] * np.asarray(kmax, dtype=np.float64)[None, :, :]
    return np.maximum(lo, hi).sum(axis=2).max(axis=0)


def quest_k_pages(budget_tokens: int, page_size: int = PAGE) -> int:
    """Pages allowed by a token budget: max(1, floor(budget / page_size))."""
    return max(1, int(budget_tokens) // page_size)


def quest_select(U, k: int) -> np.ndarray:
    """Selected logical page ids, ascending: the last page, plus the k-1 best
    of the others under (score desc, page asc); all pages when n <= k."""
    U = np.asarray(U, dtype=np.float64)
    n = len(U)
    if n <= k:
        return np.arange(n)
    others = top_k(U[:n - 1], k - 1)
    return np.concatenate([others, [n - 1]]).astype(np.int64)


def selected_tokens(pages, ctx: int, page_size: int = PAGE) -> np.ndarray:
    """Token positions covered by the selected pages (valid tokens only)."""
    out = [np.arange(p * page_size, min(ctx, (p + 1) * page_size)) for p in pages]
    return np.concatenate(out) if out else np.zeros(0, dtype=np.int64)
