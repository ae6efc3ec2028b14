"""H2O's token-level accumulate-then-evict step as a special case of the router.

Test infrastructure (see ``oracle/__init__``).

Source: H2O page (PaperTrace 3.1.2), §1.2 (capacity B = B_h + B_r with a
recent region of B_r positions) and §2.1 (order: append, attend over the
temporary candidates, add the weights to the cumulative scores, then evict
the lowest-scoring position outside the recent region).

With windows of one token, no sink, K_f = B_h, K_q = 0 and n_recent = B_r,
the tiered router performs exactly this step: the position leaving the recent
region joins the heavy hitters as a candidate and the lowest of them goes.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Sequence

import numpy as np

from .router import EVICTED, FULL, PINNED, assign, candidate_pool

F32 = np.float32


def h2o_step(heavy: Dict[int, float], recent: Dict[int, float], new_pos: int,
             weights: Sequence[float], n_heavy: int, n_recent: int):
    """One decode step of H2O with given attention weights.

    ``heavy``/``recent`` map original positions to cumulative scores before
    the step; ``weights`` are the attention weights of the new query over
    heavy + recent + [new_pos] in ascending position order.  Returns
    (scores after accumulation {pos: float32}, evicted positions, cache after
    the step as a sorted position list).
    """
    tier = {p: FULL for p in heavy}
    tier.update({p: PINNED for p in recent})
    tier[new_pos] = PINNED
    S = {p: F32(s) for p, s in {**heavy, **recent}.items()}
    S[new_pos] = F32(0)
    order = sorted(tier)
    assert len(weights) == len(order)
    for p, a in zip(order, weights):
        S[p] = F32(S[p] + F32(a))
    L = new_pos + 1
    cands = candidate_pool(tier, L, 1, n_recent)
    res = assign(cands, S, n_heavy, 0)
    for p in res.evicted:
        tier[p] = EVICTED
    cache = sorted(p for p, z in tier.items() if z != EVICTED)
    return S, res.evicted, cache
