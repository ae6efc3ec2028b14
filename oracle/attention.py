"""Decode attention over the accessible mixed-precision set.

Test infrastructure (see ``oracle/__init__``).

Sources
-------
* QEvict reading notes, §4.1 eq. "attention": a_t = softmax(q K_acc^T /
  sqrt(d)), o_t = a_t V_acc, where K_acc/V_acc are the Full windows and the
  dequantized INT2 windows; evicted windows take no part.
* H2O page, §1.1: the softmax is normalised over the candidates present at
  this step (the removed positions change the denominator).
* H2O page, §5.1 "GQA": the increment of a KV head's score is the sum over
  the query heads of its group, Delta S_{g,i} = sum_{h in g} a_{h,i}.
"""
from __future__ import annotations

import numpy as np


def softmax_attention(q, K, V):
    """q [G, d], K [n, d], V [n, d] (float64) -> (o [G, d], p [G, n])."""
    d = q.shape[1]
    logits = (q @ K.T) / np.sqrt(d)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    p = e / e.sum(axis=1, keepdims=True)
    return p @ V, p


def group_mass(p, token_window, windows):
    """Sum of p over the group's query heads and over each window's tokens.

    p [G, n]; token_window [n] window index of each accessible token (-1 for
    sink tokens, which are never scored); returns {window: float64 mass}.
    """
    col = p.sum(axis=0)
    return {j: float(col[token_window == j].sum()) for j in windows}
