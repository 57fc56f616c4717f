"""Oracle: the MoE routing cascade, pass by pass in fp64.

Test infrastructure only (see the package docstring for who may import it).

The cascade ([E] §4.2):

    scores  = x @ W_gate          (a GEMM: one dot product per token/expert)
    top_k   = TopK(scores)        (a selection reduction over experts)
    weights = softmax(top_k)      (max, sum-exp and normalise over the k
                                   selected scores only)

Readings where the article is silent: top-k is taken first and softmax runs
over the k selected scores (the order in which the article writes the
steps); the selected experts are listed by descending score, and equal
scores are ordered by ascending expert index.  W_gate is stored
expert-major, [E][D].
"""
from __future__ import annotations

import numpy as np


def _f64(t) -> np.ndarray:
    if hasattr(t, "detach"):
        import torch

        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def gate_scores(x, w_gate) -> np.ndarray:
    """scores[t, e] = sum_d x[t, d] * W_gate[e, d]  (x [T,D], W_gate [E,D])."""
    return _f64(x) @ _f64(w_gate).T


def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices [T, k] of the k best experts per token: sort by descending
    score, equal scores by ascending index (a stable sort of -score keeps
    the lower index first), keep the first k."""
    order = np.argsort(-scores, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def softmax_selected(sel: np.ndarray) -> np.ndarray:
    """Safe softmax over the selected scores of each token, [T, k]."""
    m = sel.max(axis=1, keepdims=True)
    e = np.exp(sel - m)
    return e / e.sum(axis=1, keepdims=True)


def moe_gate(x, w_gate, k: int, rows=None):
    """Returns (idx int32 [T,k], weights fp64 [T,k], scores fp64 [T,E]);
    with ``rows`` (token indices) only those tokens are computed."""
    xs = x if rows is None else x[list(rows)]
    scores = gate_scores(xs, w_gate)                        # pass 1
    idx = topk_select(scores, k)                            # pass 2
    sel = np.take_along_axis(scores, idx.astype(np.int64), axis=1)
    w = softmax_selected(sel)                               # pass 3
    return idx, w, scores
