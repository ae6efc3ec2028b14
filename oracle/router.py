"""Tier routing at a routing event.

Test infrastructure (see ``oracle/__init__``).

Sources
-------
* QEvict reading notes, §4.4 eq. (4): the candidate pool is the previous
  Full set, the previous Quantized set and the windows that have just aged
  out of the protected recent region.
* QEvict reading notes, §4.4 eq. (5) and Algorithm 1: candidates are
  sorted by cumulative score, the top K_f become Full, the next K_q
  Quantized, the rest Evicted; eq. (6): Evicted is final.
* H2O page, §5.1 and §6 ("ties"): ties are broken on the original position,
  never on the physical slot; here the lower original position (lower
  window index) ranks first.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np

PINNED, FULL, QUANT, EVICTED = "P", "F", "Q", "E"


@dataclasses.dataclass
class RouteResult:
    kf: int
    kq: int
    order: List[int]           # candidates, best first
    full: List[int]
    quant: List[int]
    evicted: List[int]
    margin_f: float            # lowest Full score minus highest non-Full score (inf if no cut)
    margin_q: float            # lowest kept score minus highest evicted score (inf if no cut)


def aged_windows(tier: Dict[int, str], L: int, window: int, n_recent: int) -> List[int]:
    """Pinned windows wholly older than the recent region [L - n_recent, L)."""
    return sorted(j for j, z in tier.items() if z == PINNED and (j + 1) * window <= L - n_recent)


def candidate_pool(tier: Dict[int, str], L: int, window: int, n_recent: int) -> List[int]:
    """eq. (4): F_{t-Omega} u Q_{t-Omega} u L_aged."""
    prev = [j for j, z in tier.items() if z in (FULL, QUANT)]
    return sorted(set(prev) | set(aged_windows(tier, L, window, n_recent)))


def rank(cands: List[int], scores: Dict[int, np.float32]) -> List[int]:
    """Sort by score descending, ties by lower window index."""
    return sorted(cands, key=lambda j: (-float(scores[j]), j))


def assign(cands: List[int], scores: Dict[int, np.float32], kf: int, kq: int) -> RouteResult:
    """eq. (5): greedy TopK_{K_f}, then TopK_{K_q} of the rest, the remainder evicted."""
    order = rank(cands, scores)
    full, quant, ev = order[:kf], order[kf:kf + kq], order[kf + kq:]

    def gap(i):
        if 0 < i < len(order):
            return float(scores[order[i - 1]]) - float(scores[order[i]])
        return float("inf")

    return RouteResult(kf, kq, order, full, quant, ev, gap(kf), gap(kf + kq))
