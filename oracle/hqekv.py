"""Five-tier per-token cache of the HqeKV kind: BF16 / INT4 / INT2 (uniform) / 1-bit (normal) /
evicted, re-ranked and re-quantized periodically, demote only.

Test infrastructure (see ``oracle/__init__``).

Sources (HqeKV reading notes, zhongzhuzhou.org, 2026-08-26)
------------------------------------------------------------
* §2.3 eq. (2): uniform quantization of a 1 x D vector with offset z = min and
  scale s = (max - min) / (2^b - 1); each value goes to the nearest level.
* §2.3 eqs. (3)-(4): normalized quantization: x' = (x - m) / s with m and s the
  vector's mean and standard deviation; the 2^b centers sit at standard normal
  quantiles; a value takes the center with the least normal probability mass
  between the two.
* §3.1: five actions per cached pair (FP16, 4-bit, 2-bit, 1-bit, evict); 4- and
  2-bit tiers quantize uniformly, the 1-bit tier with the normal quantizer (§3.4).
* §3.2: the key importance is the cumulative attention weight; the joint value
  metric multiplies it by the token's value range.
* §3.3, §3.7: fixed fractions applied to the importance ranking (the search that
  picks the fractions runs offline and is not part of the decode path).
* §3.5, §3.8: every T tokens the cache is re-ranked and re-quantized; a token
  only ever moves to a lower precision.
* §3.10: the cumulative attention is counted over the most recent m queries
  (m = 20).

Readings where the pages leave a step open
------------------------------------------
* Groups are per token: one (z, s) or (m, s) pair for a token's key and one for
  its value, over the head dimension.
* Normal centers c_j = Phi^-1((j + 1/2) / 2^b), j = 0 .. 2^b - 1 (the printed
  index range is garbled); the decision boundary between c_j and c_(j+1) is
  Phi^-1((j + 1) / 2^b), where the two probability masses are equal, and a
  value on a boundary takes the lower center.  For b = 1 the centers are
  +-0.6745 and the boundary is 0: the code is 1 exactly when x > m.
* Mean and population standard deviation (eq. (3)) are the exact values for the
  token's float32 entries, each rounded once to the nearest float32 (ties to even): m =
  round(sum x / D), s = round(sqrt(sum (x - mean)^2 / D)) with the exact mean inside the
  square.  The pages fix neither a precision nor an order of summation; exact values
  rounded once depend on neither.  s = 0 gives all-zero codes.
* Uniform decisions are eq. (2) in float32 as in ``oracle.quant``.
* Dequantization is one float32 fused multiply-add, code * s + z (uniform) or
  c_j * s + m (normal); re-quantization to a lower tier starts from those
  values, since no higher-precision copy is kept (§3.5).  A token whose tier
  does not change keeps its codes.
* Fractions are of the current length L; the BF16 share includes the sink and
  recent tokens, which are never ranked: n_bf16 = max(0, floor(f_bf16 L) -
  n_sink - n_recent), n_b = floor(f_b L) for the other tiers, the rest evicted.
* Ranking: importance descending, ties to the lower position; a token's new tier
  is the lower of its current tier and the one its rank gives.
* Scores: each decode step adds, to every accessible non-sink token, the
  attention mass summed over the KV head's query heads (float64, rounded once
  to float32 and added to the float32 score), but only on the last m steps
  before a re-rank (m = 0: every step); scores restart at 0 after each re-rank
  when m > 0.
* Prefill tokens start BF16 with score 0; the first re-rank is at decode step T.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from .attention import softmax_attention
from .quant import uniform_quantize

F32 = np.float32

BF16, INT4, INT2, NQ1, EVICT = 0, 1, 2, 3, 4
TIER_NAMES = ("bf16", "int4", "int2", "nq1", "evicted")
TIER_BITS = {INT4: 4, INT2: 2, NQ1: 1}


# --------------------------------------------------------------------------- exact float32 fma
def fmaf32(a, b, c):
    """float32(a * b + c) rounded once, for float32 arrays (what the CUDA fmaf returns).

    a * b is exact in float64 (24 + 24 bits); s = ab + c is rounded to float64 and its
    error e recovered exactly (Knuth's TwoSum), so the exact result is s + e.  Rounding s
    to float32 gives the right answer unless s lies exactly halfway between two float32
    neighbours and e is not zero; then the exact result is on e's side of that midpoint.
    """
    a = np.asarray(a, np.float32).astype(np.float64)
    b = np.asarray(b, np.float32).astype(np.float64)
    c = np.asarray(c, np.float32).astype(np.float64)
    p = a * b
    s = p + c
    bb = s - p
    e = (p - (s - bb)) + (c - bb)
    r = np.asarray(s.astype(np.float32))
    r64 = r.astype(np.float64)
    up = np.nextafter(r, np.float32(np.inf))
    dn = np.nextafter(r, np.float32(-np.inf))
    below = s == (r64 + dn.astype(np.float64)) / 2     # the tie was rounded up to r
    above = s == (r64 + up.astype(np.float64)) / 2     # the tie was rounded down to r
    r = np.where(below & (e < 0), dn, r)
    r = np.where(above & (e > 0), up, r)
    return r.astype(np.float32)


# --------------------------------------------------------------------------- standard normal
def normal_cdf(x):
    """Phi(x) in float64 from the complementary error function."""
    x = np.asarray(x, np.float64)
    return 0.5 * np.vectorize(math.erfc)(-x / math.sqrt(2.0))


def normal_ppf(p: float) -> float:
    """Phi^-1(p) by Newton's method on Phi(x) - p (Phi from erfc), float64."""
    if p == 0.5:
        return 0.0
    x = 0.0
    for _ in range(200):
        f = 0.5 * math.erfc(-x / math.sqrt(2.0)) - p
        dens = math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)
        step = f / dens
        x -= step
        if abs(step) <= 1e-17 * max(1.0, abs(x)):
            break
    return x


def _symmetric(points: List[float]) -> np.ndarray:
    """Phi^-1 at the given probabilities, the lower half mirrored from the upper half
    (Phi^-1(1 - p) = -Phi^-1(p))."""
    n = len(points)
    out = np.zeros(n, np.float64)
    for j in range(n):
        jj = n - 1 - j
        if points[j] >= 0.5:
            out[j] = normal_ppf(points[j])
        else:
            out[j] = -normal_ppf(points[jj])
    return out


def normal_centers(bits: int) -> np.ndarray:
    """c_j = Phi^-1((j + 1/2) / 2^b) as float64."""
    n = 1 << bits
    return _symmetric([(j + 0.5) / n for j in range(n)])


def normal_boundaries(bits: int) -> np.ndarray:
    """Equal-mass points between neighbouring centers, Phi^-1((j + 1) / 2^b)."""
    n = 1 << bits
    return _symmetric([(j + 1) / n for j in range(n - 1)])


def _f32_exp_floor(num: int, den: int) -> int:
    """floor(log2(num / den)) for integers num, den > 0."""
    e = num.bit_length() - den.bit_length()
    if (num << max(0, -e)) < (den << max(0, e)):
        e -= 1
    return e


def _f32_from_ratio(num: int, den: int) -> np.float32:
    """num / den (integers, den > 0) rounded to the nearest float32, ties to even, with
    subnormals (the spacing of float32 values below 2^-126 is 2^-149)."""
    if num == 0:
        return F32(0.0)
    a = abs(num)
    q = max(_f32_exp_floor(a, den) - 23, -149)          # exponent of the result's last place
    n, r = divmod(a << -q, den) if q < 0 else divmod(a, den << q)
    rd = den if q < 0 else den << q
    if 2 * r > rd or (2 * r == rd and n & 1):
        n += 1
    v = F32(math.ldexp(n, q))                              # exact: n <= 2^24
    return -v if num < 0 else v


def _f32_sqrt_of_ratio(num: int, den: int) -> np.float32:
    """sqrt(num / den) (integers, num >= 0, den > 0) rounded to the nearest float32, ties to
    even: n = floor(sqrt(y)) for y = num / (den 4^q) from an integer square root, then one
    exact comparison of y with (n + 1/2)^2."""
    if num == 0:
        return F32(0.0)
    q = max(_f32_exp_floor(num, den) // 2 - 23, -149)
    if q < 0:
        ynum, yden = num << (-2 * q), den
    else:
        ynum, yden = num, den << (2 * q)
    n = math.isqrt(ynum // yden)
    lhs, rhs = 4 * ynum, (4 * n * n + 4 * n + 1) * yden    # y vs (n + 1/2)^2, times 4 yden
    if lhs > rhs or (lhs == rhs and n & 1):
        n += 1
    return F32(math.ldexp(n, q))


def mean_std_f32(x):
    """Per-row mean and population std of x [n, D] (float32), each the exact value rounded
    once to float32 (ties to even).  Every float32 is an integer multiple of 2^-149, so with
    X_i = x_i 2^149, S = sum X_i and Q = sum X_i^2 (exact integers):
    mean = S / (D 2^149) and std = sqrt((D Q - S^2) / (D^2 2^298))."""
    x = np.asarray(x, np.float32)
    n, D = x.shape
    ints = np.ldexp(x.astype(np.float64), 149)             # exact: integers below 2^277
    m = np.zeros(n, np.float32)
    sd = np.zeros(n, np.float32)
    for r in range(n):
        X = [int(v) for v in ints[r]]
        S = sum(X)
        Q = sum(v * v for v in X)
        m[r] = _f32_from_ratio(S, D << 149)
        sd[r] = _f32_sqrt_of_ratio(D * Q - S * S, (D * D) << 298)
    return m, sd


def normal_quantize(x, bits: int = 1):
    """eqs. (3)-(4) per row of x [n, D] (float32): (codes uint8 [n, D], m float32 [n], s float32 [n])."""
    m, s = mean_std_f32(x)
    x = np.asarray(x, np.float32).astype(np.float64)
    safe = np.where(s == 0, 1.0, s.astype(np.float64))
    xp = (x - m.astype(np.float64)[:, None]) / safe[:, None]          # eq. (3)
    codes = np.zeros(x.shape, np.uint8)
    for beta in normal_boundaries(bits):                               # eq. (4): nearest in mass
        codes += (xp > beta).astype(np.uint8)
    codes[s == 0] = 0
    return codes, m, s


def normal_dequantize(codes, m, s, bits: int = 1):
    """x = c_j * s + m, one float32 fma per value."""
    c = normal_centers(bits).astype(F32)[np.asarray(codes, np.int64)]
    return fmaf32(c, np.asarray(s, F32)[:, None], np.asarray(m, F32)[:, None])


def uniform_quantize_rows(x, bits: int):
    """eq. (2) per row (token): (codes [n, D], z [n], s [n])."""
    codes, z, s = uniform_quantize(x, bits, axis=1)
    return codes, z[:, 0], s[:, 0]


def uniform_dequantize_rows(codes, z, s):
    """x = code * s + z, one float32 fma per value."""
    return fmaf32(np.asarray(codes, F32), np.asarray(s, F32)[:, None], np.asarray(z, F32)[:, None])


# --------------------------------------------------------------------------- one token's payload
@dataclasses.dataclass
class TokenCodes:
    """Codes of one token's key and value in a quantized tier, with their float32 parameters:
    (min, scale) for the uniform tiers, (mean, std) for the normal tier."""
    tier: int
    k_codes: np.ndarray
    k_p0: np.float32
    k_p1: np.float32
    v_codes: np.ndarray
    v_p0: np.float32
    v_p1: np.float32


def quantize_token(tier: int, k, v) -> TokenCodes:
    """Quantize one token (float32 [D] key and value) into a quantized tier."""
    k = np.asarray(k, F32)[None, :]
    v = np.asarray(v, F32)[None, :]
    if tier == NQ1:
        kc, k0, k1 = normal_quantize(k, 1)
        vc, v0, v1 = normal_quantize(v, 1)
    else:
        kc, k0, k1 = uniform_quantize_rows(k, TIER_BITS[tier])
        vc, v0, v1 = uniform_quantize_rows(v, TIER_BITS[tier])
    return TokenCodes(tier, kc[0], F32(k0[0]), F32(k1[0]), vc[0], F32(v0[0]), F32(v1[0]))


def dequantize_token(tc: TokenCodes) -> Tuple[np.ndarray, np.ndarray]:
    """(key, value) float32 [D] as the tier reconstructs them."""
    if tc.tier == NQ1:
        k = normal_dequantize(tc.k_codes[None, :], [tc.k_p0], [tc.k_p1])[0]
        v = normal_dequantize(tc.v_codes[None, :], [tc.v_p0], [tc.v_p1])[0]
    else:
        k = uniform_dequantize_rows(tc.k_codes[None, :], [tc.k_p0], [tc.k_p1])[0]
        v = uniform_dequantize_rows(tc.v_codes[None, :], [tc.v_p0], [tc.v_p1])[0]
    return k, v


# --------------------------------------------------------------------------- ranking
def tier_counts(L: int, n_sink: int, n_recent: int, fractions: Sequence[float]) -> Tuple[int, int, int, int]:
    """Ranked tokens per tier (BF16, INT4, INT2, 1-bit) at length L; the rest are evicted."""
    fb, f4, f2, f1 = (float(f) for f in fractions)
    nb = max(0, math.floor(fb * L) - n_sink - n_recent)
    return nb, math.floor(f4 * L), math.floor(f2 * L), math.floor(f1 * L)


def joint_metric(attention, value_range):
    """§3.2: the value importance, cumulative attention times the token's value range."""
    return np.asarray(attention, np.float64) * np.asarray(value_range, np.float64)


def rank_tiers(importance, positions, counts: Sequence[int]) -> np.ndarray:
    """Tier each token's rank gives: importance descending, ties to the lower position;
    the first counts[0] BF16, the next counts[1] INT4, counts[2] INT2, counts[3] 1-bit, rest evicted."""
    importance = np.asarray(importance)
    positions = np.asarray(positions)
    order = np.lexsort((positions, -importance.astype(np.float64)))
    tiers = np.full(len(order), EVICT, np.int64)
    start = 0
    for z, n in zip((BF16, INT4, INT2, NQ1), counts):
        tiers[order[start:start + n]] = z
        start += n
    return tiers


# --------------------------------------------------------------------------- one unit
@dataclasses.dataclass
class RerankResult:
    L: int
    counts: Tuple[int, int, int, int]
    desired: Dict[int, int]
    changed: Dict[int, Tuple[int, int]]      # position -> (old tier, new tier)


class HqeUnit:
    """Cache state of one (batch element, layer, KV head) in the five-tier per-token variant."""

    def __init__(self, head_dim: int, group: int, n_sink: int, n_recent: int, period: int,
                 score_window: int, fractions: Sequence[float], max_context: int):
        assert 0 <= score_window <= period
        self.d, self.G = head_dim, group
        self.n_sink, self.n_recent = n_sink, n_recent
        self.T, self.m = period, score_window
        self.fractions = tuple(float(f) for f in fractions)
        self.K = np.zeros((max_context, head_dim), F32)     # original bf16 values
        self.V = np.zeros((max_context, head_dim), F32)
        self.L = 0
        self.t = 0
        self.tier = np.zeros(max_context, np.int64)          # BF16 for every position at first
        self.S = np.zeros(max_context, F32)
        self.codes: Dict[int, TokenCodes] = {}
        self._deq: Dict[int, Tuple[np.ndarray, np.ndarray]] = {}
        self.history: List[RerankResult] = []

    def append(self, k_rows, v_rows):
        k_rows = np.asarray(k_rows, F32).reshape(-1, self.d)
        v_rows = np.asarray(v_rows, F32).reshape(-1, self.d)
        n = k_rows.shape[0]
        self.K[self.L:self.L + n] = k_rows
        self.V[self.L:self.L + n] = v_rows
        self.tier[self.L:self.L + n] = BF16
        self.S[self.L:self.L + n] = 0
        self.L += n

    def values(self, p: int) -> Tuple[np.ndarray, np.ndarray]:
        """Key and value of position p as its tier holds them (float32)."""
        z = self.tier[p]
        if z == BF16:
            return self.K[p], self.V[p]
        if p not in self._deq:
            self._deq[p] = dequantize_token(self.codes[p])
        return self._deq[p]

    def accessible(self):
        pos = [p for p in range(self.L) if self.tier[p] != EVICT]
        K = np.zeros((len(pos), self.d), np.float64)
        V = np.zeros((len(pos), self.d), np.float64)
        for i, p in enumerate(pos):
            k, v = self.values(p)
            K[i], V[i] = k, v
        return np.array(pos, np.int64), K, V

    def scoring_step(self, t: int) -> bool:
        """Whether decode step t (1-based) adds to the scores."""
        return self.m == 0 or (t - 1) % self.T >= self.T - self.m

    def decode_step(self, q, k_row, v_row, auto_rerank: bool = True):
        """append -> attend -> (scoring steps) accumulate -> (every T steps, when auto_rerank)
        re-rank.

        Returns (o [G, d] float64, mass {position: float64} of this step)."""
        self.append(k_row, v_row)
        self.t += 1
        pos, K, V = self.accessible()
        o, p = softmax_attention(np.asarray(q, np.float64), K, V)
        col = p.sum(axis=0)
        mass = {int(q_): float(col[i]) for i, q_ in enumerate(pos) if q_ >= self.n_sink}
        if self.scoring_step(self.t):
            for q_, mval in mass.items():
                self.S[q_] = F32(self.S[q_] + F32(mval))
        if auto_rerank and self.t % self.T == 0:
            self.rerank()
        return o, mass

    def rerank(self) -> RerankResult:
        L = self.L
        counts = tier_counts(L, self.n_sink, self.n_recent, self.fractions)
        cand = np.array([p for p in range(self.n_sink, L - self.n_recent) if self.tier[p] != EVICT], np.int64)
        desired = rank_tiers(self.S[cand], cand, counts) if len(cand) else np.zeros(0, np.int64)
        changed = {}
        for p, zd in zip(cand.tolist(), desired.tolist()):
            z0 = int(self.tier[p])
            zn = max(z0, zd)                        # demote only
            if zn == z0:
                continue
            changed[p] = (z0, zn)
            if zn == EVICT:
                self.codes.pop(p, None)
            else:
                k, v = self.values(p)               # re-quantize what the token holds now
                self.codes[p] = quantize_token(zn, k, v)
            self._deq.pop(p, None)
            self.tier[p] = zn
        if self.m > 0:
            self.S[:L] = 0
        res = RerankResult(L, counts, dict(zip(cand.tolist(), desired.tolist())), changed)
        self.history.append(res)
        return res

    def tier_histogram(self) -> Tuple[int, ...]:
        return tuple(int(np.sum(self.tier[:self.L] == z)) for z in range(5))
