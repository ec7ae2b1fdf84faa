"""SnapKV observation-window scoring, pooling, selection and compaction (oracle).

SnapKV looks at how the last few query rows attend to the history, keeps the
important part and physically deletes the rest ("tokendh.com article",
section "把边界划在'生命周期'上"); a retained token keeps its logical
position even though its storage moves ("tokendh.com article", section
"聊天记录也能'续命':Chain Cache").

Definitions used here (for one sequence and one KV head):

* window rows: the last W query rows (positions L-W .. L-1), each with the G
  query heads of the KV head's group;
* row i, head g attends causally: keys j <= L-W+i, p = softmax_j(scale*q.k_j)
  over exactly those keys (prefix, earlier window keys and itself);
* column score A[j] = sum over rows i and heads g of p[i,g,j];
* selection: max-pool A over the candidate prefix [0, L-R) with a stride-1,
  same-length window of ``kernel`` (out-of-range neighbours ignored); keep the
  best ``keep`` candidates under (pooled score desc, position asc), plus the
  R most recent positions [L-R, L); SnapKV uses R = W; if L-R <= keep all
  candidates are kept;
* compaction: the kept rows of K and V, ascending position, with their
  logical positions.
"""
import numpy as np

from .topk import top_k


def window_scores(q_win, k, scale: float):
    """A[j] for all L key positions.  q_win [W][G][D] holds the query rows of
    positions L-W..L-1 (for the KV head's G query heads); k [L][D]."""
    q = np.asarray(q_win, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    W, G, _ = q.shape
    L = k.shape[0]
    A = np.zeros(L)
    for i in range(W):
        last = L - W + i                      # this row's own position
        s = scale * (q[i] @ k[:last + 1].T)   # [G][last+1]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / e.sum(axis=1, keepdims=True)
        A[:last + 1] += p.sum(axis=0)
    return A


def max_pool(a, kernel: int):
    """Stride-1 max-pool with an odd window, same length, borders clipped."""
    a = np.asarray(a, dtype=np.float64)
    if kernel % 2 != 1:
        raise ValueError("pool kernel must be odd")
    r = kernel // 2
    n = len(a)
    out = np.empty(n)
    for j in range(n):
        out[j] = a[max(0, j - r):min(n, j + r + 1)].max()
    return out


def keep_positions(A, L: int, recent: int, keep: int, kernel: int):
    """Kept positions (ascending): top-``keep`` of the pooled candidate scores
    over [0, L-recent) plus the ``recent`` newest positions."""
    A = np.asarray(A, dtype=np.float64)
    n_cand = max(0, L - recent)
    pooled = max_pool(A[:n_cand], kernel) if n_cand else np.zeros(0)
    chosen = top_k(pooled, keep)
    return np.concatenate([chosen, np.arange(n_cand, L)]).astype(np.int64)


def compact(k, v, positions):
    """Rows of k and v at ``positions`` (ascending) and the positions."""
    pos = np.asarray(positions, dtype=np.int64)
    return np.asarray(k)[pos], np.asarray(v)[pos], pos
