"""Writes the golden fixtures of this directory from the oracle alone.

Inputs are small, explicit and exactly representable in bfloat16 (multiples of
1/4 in [-2, 2]); expected values are the oracle's (oracle/ only, float64).
Definitions: Quest page selection (tokendh.com article on SparseEngine,
section "历史太长,会撑爆什么"), SnapKV window scores and H2O accumulated
scores (same article, section "把边界划在'生命周期'上").

    python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def quarter_grid(g, shape):
    return (g.integers(-8, 9, size=shape) / 4.0).astype(np.float64)


def quest_case():
    g = np.random.default_rng(20261202)
    D, G, T, budget = 64, 2, 40, 32
    k, v, q = quarter_grid(g, (T, D)), quarter_grid(g, (T, D)), quarter_grid(g, (G, D))
    kmin, kmax = oracle.page_minmax(k)
    U = oracle.quest_bound(q, kmin, kmax)
    pages = oracle.quest_select(U, oracle.quest_k_pages(budget))
    tok = oracle.quest.selected_tokens(pages, T)
    out, lse = oracle.attend(q, k[tok], v[tok], 1 / math.sqrt(D))
    return {"what": "Quest: 1 sequence, 2 query heads / 1 KV head, D=64, 40 tokens, budget 32",
            "head_dim": D, "group": G, "ctx": T, "budget": budget,
            "k": k.tolist(), "v": v.tolist(), "q": q.tolist(),
            "expected": {"U": U.tolist(), "pages": pages.tolist(), "out": out.tolist(),
                         "lse": lse.tolist()}}


def snapkv_case():
    g = np.random.default_rng(20261203)
    D, G, L, W, pool, keep = 64, 2, 40, 4, 3, 8
    k, v, qw = quarter_grid(g, (L, D)), quarter_grid(g, (L, D)), quarter_grid(g, (W, G, D))
    A = oracle.window_scores(qw, k, 1 / math.sqrt(D))
    kept = oracle.keep_positions(A, L, W, keep, pool)
    return {"what": "SnapKV: 1 sequence, 2 query heads / 1 KV head, D=64, L=40, window 4, "
                    "pool 3, keep 8",
            "head_dim": D, "group": G, "ctx": L, "window": W, "pool": pool, "keep": keep,
            "k": k.tolist(), "v": v.tolist(), "q_win": qw.tolist(),
            "expected": {"A": A.tolist(), "kept": kept.tolist()}}


def h2o_case():
    g = np.random.default_rng(20261204)
    D, G, n, budget, recent = 64, 2, 12, 12, 2
    pos = np.array([0, 1, 2, 3, 5, 8, 9, 13, 14, 17, 18, 19])
    k, v = quarter_grid(g, (n, D)), quarter_grid(g, (n, D))
    score = (g.integers(0, 40, size=n) / 8.0).astype(np.float64)
    q, kn, vn = quarter_grid(g, (G, D)), quarter_grid(g, (D,)), quarter_grid(g, (D,))
    st = oracle.H2OState(pos=pos.copy(), k=k, v=v, score=score.copy())
    new, out, lse, ev = oracle.h2o_step(st, q, kn, vn, 20, budget, recent, 1 / math.sqrt(D))
    order = np.argsort(new.pos)
    return {"what": "H2O: one step, 12 held tokens, budget 12, recent 2, new position 20",
            "head_dim": D, "group": G, "budget": budget, "recent": recent, "new_pos": 20,
            "pos": pos.tolist(), "k": k.tolist(), "v": v.tolist(), "score": score.tolist(),
            "q": q.tolist(), "k_new": kn.tolist(), "v_new": vn.tolist(),
            "expected": {"evicted": ev, "out": out.tolist(), "lse": lse.tolist(),
                         "pos_after": new.pos[order].tolist(),
                         "score_after": new.score[order].tolist()}}


def main():
    for name, fn in (("quest_tiny", quest_case), ("snapkv_tiny", snapkv_case),
                     ("h2o_tiny", h2o_case)):
        case = fn()
        case["source"] = "written by tests/golden/make_golden.py from oracle/ (float64)"
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(case, f, indent=None, separators=(",", ":"))
        print(name, "ok")


if __name__ == "__main__":
    main()
