"""Comparison rules between the CUDA path and the oracle.

Indices: exact, except that a page/position chosen by one side and not the
other is allowed when its oracle score lies within 1e-5 (relative) of the
oracle's boundary score (the k-th best).  Outputs: max-abs error 2e-2 for bf16
outputs, 1e-3 for fp32 outputs.
"""
import numpy as np

REL_BOUNDARY = 1e-5
TOL_BF16 = 2e-2
TOL_F32 = 1e-3


def bf16_tensor_to_f64(t):
    """A torch bf16/f32 tensor (any device) as float64 numpy."""
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def check_topk(gpu_idx, ora_idx, scores, k_boundary, rel=REL_BOUNDARY, what="selection"):
    """gpu_idx / ora_idx: selected indices (any order); scores: oracle scores
    indexed by those indices; k_boundary: the oracle's k-th best score.
    Returns the number of allowed mismatches; raises AssertionError otherwise."""
    g, o = set(int(x) for x in gpu_idx), set(int(x) for x in ora_idx)
    assert len(g) == len(o), f"{what}: sizes differ ({len(g)} vs {len(o)})"
    diff = g ^ o
    tol = rel * max(abs(k_boundary), 1e-30)
    bad = [i for i in diff if abs(scores[i] - k_boundary) > tol]
    assert not bad, (f"{what}: {len(bad)} mismatches outside the boundary allowance, e.g. "
                     f"{bad[:5]} scores {[scores[i] for i in bad[:5]]} boundary {k_boundary}")
    return len(diff) // 2


def max_abs(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0
