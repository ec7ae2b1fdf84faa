"""Span-restricted prefix pruning and the StreamingLLM view (oracle).

Prefix-cache pruning lets the application name a region of the history and
how much of it to keep; a scorer picks the tokens of the region worth
keeping and the rest is deleted, while the logical prefix stays whole for
prefix matching ("tokendh.com article", section "该删哪段历史,让应用自己说了算:
可控前缀裁剪"; "SparseEngine 统一接入十五种稀疏注意力", section "Agent 轨迹、Chain Cache
与 prefix pruning": keep 20% of the aligned KV tokens of chosen tool results).
StreamingLLM (named among the compared methods, same page, section "哪些情况下
加速幅度会缩小") keeps the first tokens and a recent window.

Definitions used here (one sequence, one KV head):

* span pruning: candidates are the positions [s0, s1) of the span (clipped
  to [0, L)); their scores are the SnapKV window column scores
  (``snapkv.window_scores``; the pages name KVzip as a scorer but do not
  describe it -- a reading), max-pooled over the span with the odd window
  ``kernel`` (neighbours outside the span ignored); the best ``keep``
  candidates under (pooled desc, position asc) are kept; every position
  outside the span is kept; the kept positions are ascending and stay the
  tokens' logical positions;
* sink + recent view: the pages [0, sink_pages) and the last ``recent_pages``
  pages of the sequence (pages of 16 tokens; a reading at page granularity,
  the view's unit), all pages when they overlap; attention over their valid
  tokens.
"""
import numpy as np

from .snapkv import max_pool
from .topk import top_k

PAGE = 16


def span_keep_positions(A, L: int, s0: int, s1: int, keep: int, kernel: int) -> np.ndarray:
    """Kept positions of a sequence of L tokens whose span [s0, s1) is pruned
    to its best ``keep`` tokens by the pooled scores A[s0:s1]."""
    A = np.asarray(A, dtype=np.float64)
    s0 = max(0, min(int(s0), L))
    s1 = max(s0, min(int(s1), L))
    cand = np.zeros(0, dtype=np.int64)
    if s1 > s0:
        pooled = max_pool(A[s0:s1], kernel)
        cand = top_k(pooled, keep) + s0
    return np.concatenate([np.arange(s0), cand, np.arange(s1, L)]).astype(np.int64)


def sink_recent_pages(L: int, sink_pages: int, recent_pages: int) -> np.ndarray:
    """Pages of the sink + recent view of a sequence of L tokens, ascending."""
    n = -(-int(L) // PAGE)
    first = np.arange(min(int(sink_pages), n))
    last = np.arange(max(min(int(sink_pages), n), n - int(recent_pages)), n)
    return np.concatenate([first, last]).astype(np.int64)
