"""Per-(batch, layer, KV head) state machine of the tiered cache.

Test infrastructure (see ``oracle/__init__``).

Sources
-------
* QEvict reading notes, §2 Figure 1: the history is cut into contiguous
  windows, all of which start in full precision; sink and recent tokens stay
  full precision.
* QEvict reading notes, §4.1: a protected sink prefix S and recent region
  L_t are never routed; every other window is Full, Quantized or Evicted.
* QEvict reading notes, §4.2 eq. (1): window scores are additive sums of the
  attention mass received, never decayed.
* QEvict reading notes, §4.4 eqs. (4)-(6) and Algorithm 1: routing every
  Omega tokens; quantize on first demotion only and reuse the ledger codes;
  Evicted is final.
* H2O page, §2.1: per-step order append -> attention over the current
  candidates (including the new token) -> score update -> eviction.

Readings where the pages leave a step open:
* window j covers positions [j w, (j+1) w); the sink tokens are carved out of
  window 0, whose routable part is [n_sink, w);
* a window is "Pinned" (full precision, not ranked) until it is complete and
  wholly older than the recent region [L - n_recent, L); at the next routing
  event it enters the candidate pool (eq. (4)'s L_aged);
* every accessible non-sink token adds to its window's score, pinned ones
  included (H2O's recent tokens are scored from their first step);
* the score increment of a KV head is the sum over its query heads;
* promotion restores the original bf16 values exactly (they are kept in a
  host backing store); keys carry no rotary embedding in these workloads,
  so no re-rotation step applies.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Tuple

import numpy as np

from .attention import group_mass, softmax_attention
from .quant import QuantizedWindow, kivi_quantize_window
from .rope import apply_rope
from .router import EVICTED, FULL, PINNED, QUANT, RouteResult, assign, candidate_pool

F32 = np.float32


class QEvictUnit:
    """Cache state of one (batch element, layer, KV head)."""

    def __init__(self, window: int, n_sink: int, n_recent: int, head_dim: int, group: int,
                 capacity: Callable[[int], Tuple[int, int]], max_context: int,
                 v_group: Optional[int] = None, rope_base: float = 0.0):
        """rope_base > 0: keys are stored pre-RoPE and rotated at their original positions when
        attended to (``oracle.rope``)."""
        assert 0 <= n_sink < window
        self.w, self.n_sink, self.n_recent = window, n_sink, n_recent
        self.d, self.G = head_dim, group
        self.v_group = head_dim if v_group is None else v_group
        self.capacity = capacity
        self.K = np.zeros((max_context, head_dim), dtype=F32)   # original bf16 values
        self.V = np.zeros((max_context, head_dim), dtype=F32)
        self.L = 0
        self.t = 0                                              # decode steps done
        self.tier: Dict[int, str] = {}
        self.S: Dict[int, np.float32] = {}
        self.ledger: Dict[int, QuantizedWindow] = {}
        self._deq: Dict[int, Tuple[np.ndarray, np.ndarray]] = {}
        self.history: List[RouteResult] = []
        self.rope_base = float(rope_base)

    # ------------------------------------------------------------------ geometry
    def window_range(self, j: int) -> Tuple[int, int]:
        """Valid positions [lo, hi) of window j at the current length."""
        lo = self.n_sink if j == 0 else j * self.w
        return lo, min((j + 1) * self.w, self.L)

    # ------------------------------------------------------------------ append
    def append(self, k_rows, v_rows):
        """Write new tokens (bf16 values as float32 [n, d]); new windows start Pinned."""
        k_rows = np.asarray(k_rows, F32).reshape(-1, self.d)
        v_rows = np.asarray(v_rows, F32).reshape(-1, self.d)
        n = k_rows.shape[0]
        self.K[self.L:self.L + n] = k_rows
        self.V[self.L:self.L + n] = v_rows
        for p in range(self.L, self.L + n):
            j = p // self.w
            if j not in self.tier:
                self.tier[j] = PINNED
                self.S[j] = F32(0)
        self.L += n

    # ------------------------------------------------------------------ attention
    def dequantized(self, j: int):
        if j not in self._deq:
            self._deq[j] = self.ledger[j].dequantize()
        return self._deq[j]

    def accessible(self):
        """(K_acc, V_acc, window of each token): sink, Pinned/Full originals, dequantized INT2."""
        ks, vs, ws, ps = [], [], [], []
        ns = min(self.n_sink, self.L)
        ks.append(self.K[:ns].astype(np.float64))
        ps.append(np.arange(ns))
        vs.append(self.V[:ns].astype(np.float64))
        ws.append(np.full(ns, -1))
        for j in sorted(self.tier):
            z = self.tier[j]
            lo, hi = self.window_range(j)
            if hi <= lo or z == EVICTED:
                continue
            if z in (PINNED, FULL):
                k, v = self.K[lo:hi].astype(np.float64), self.V[lo:hi].astype(np.float64)
            else:
                k, v = self.dequantized(j)
            ks.append(k)
            vs.append(v)
            ws.append(np.full(hi - lo, j))
            ps.append(np.arange(lo, hi))
        K = np.concatenate(ks)
        if self.rope_base > 0:                   # pre-RoPE keys, rotated at their original positions
            K = apply_rope(K, np.concatenate(ps), self.rope_base)
        return K, np.concatenate(vs), np.concatenate(ws)

    def attend(self, q):
        """Attention of the group's queries q [G, d] over the accessible set.

        Returns (o [G, d] float64, {window: group mass float64}, sink mass).
        """
        K, V, tw = self.accessible()
        o, p = softmax_attention(np.asarray(q, np.float64), K, V)
        live = [j for j, z in self.tier.items() if z != EVICTED]
        mass = group_mass(p, tw, live)
        sink_mass = float(p[:, tw == -1].sum())
        return o, mass, sink_mass

    def accumulate(self, mass: Dict[int, float]):
        """eq. (1) with the GQA group sum: S[j] += mass[j], stored in float32."""
        for j, m in mass.items():
            self.S[j] = F32(self.S[j] + F32(m))

    def decode_step(self, q, k_row, v_row):
        """append -> attend -> accumulate; returns (o, mass, sink_mass)."""
        self.append(k_row, v_row)
        o, mass, sink_mass = self.attend(q)
        self.accumulate(mass)
        self.t += 1
        return o, mass, sink_mass

    # ------------------------------------------------------------------ speculative verify
    def verify(self, qs, k_rows, v_rows):
        """Draft tokens j = 0 .. n-1 are appended one by one and query j attends over the cache
        and drafts 0 .. j; the masses are held back (H2O page §5, speculative decoding: a
        rejected draft's score increments must not reach the scores).  Returns ([o_j], [mass_j])."""
        n = len(qs)
        self._verify = (self.L, n, [])
        outs = []
        for j in range(n):
            self.append(k_rows[j], v_rows[j])
            o, mass, _ = self.attend(qs[j])
            outs.append(o)
            self._verify[2].append(mass)
        return outs, list(self._verify[2])

    def commit(self, n_accept: int):
        """Keep drafts 0 .. n_accept-1: the length becomes L0 + n_accept, windows opened by rejected
        drafts close, and the accepted queries' masses are added in order (eq. (1), float32)."""
        L0, n, masses = self._verify
        assert 0 <= n_accept <= n
        new_L = L0 + n_accept
        last = (new_L + self.w - 1) // self.w          # windows [0, last) hold a token
        for j in sorted(self.tier, reverse=True):
            if j >= last and j * self.w >= L0:           # opened by a rejected draft
                del self.tier[j]
                self.S.pop(j, None)
        self.L = new_L
        for m in masses[:n_accept]:
            self.accumulate(m)
        self.t += n_accept
        self._verify = None

    # ------------------------------------------------------------------ routing
    def quantize_window(self, j: int) -> QuantizedWindow:
        lo, hi = self.window_range(j)
        return kivi_quantize_window(self.K[lo:hi], self.V[lo:hi], bits=2, v_group=self.v_group)

    def route(self) -> RouteResult:
        """Algorithm 1 at the current length."""
        kf, kq = self.capacity(self.L)
        cands = candidate_pool(self.tier, self.L, self.w, self.n_recent)
        res = assign(cands, self.S, kf, kq)
        for j in res.quant:
            if j not in self.ledger:              # first demotion: quantize once
                self.ledger[j] = self.quantize_window(j)
            self.tier[j] = QUANT                  # later demotions reuse the ledger codes
        for j in res.full:
            self.tier[j] = FULL                   # promotion restores the original bf16
        for j in res.evicted:
            self.tier[j] = EVICTED                # final
            self.ledger.pop(j, None)
            self._deq.pop(j, None)
        self.history.append(res)
        return res
