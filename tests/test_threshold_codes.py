"""The 2-bit code rule the pack kernel applies (HqeKV reading notes, eq. (2) with b = 2):
code = rint(q) clamped to [0, 3], with q = fl(d / s) the float32 quotient and rint rounding
half to even.

For q >= 0 that code equals [q > 1/2] + [q >= 3/2] + [q > 5/2]: a quotient of exactly 1/2
rounds to 0, 3/2 to 2 and 5/2 to 2.  fl(d / s) never decreases as d grows, so each term is
[d >= T] for the smallest float32 T that passes it.  The kernel finds each T with a few
correctly rounded divisions next to fl(t s) and then compares.  This test restates that
search in numpy float32 (IEEE division) and checks it against the division, element by
element, over scales from 1e-30 to 1e30 and at every boundary and its neighbours.
"""
import numpy as np

F32 = np.float32


def code_by_division(d: np.ndarray, s: np.float32) -> np.ndarray:
    if s == 0:
        return np.zeros(d.shape, np.int64)
    q = np.rint(d.astype(F32) / F32(s))
    return np.clip(q, 0, 3).astype(np.int64)


def smallest_passing(s: np.float32, t: float, strict: bool) -> np.float32:
    """Smallest non-negative float32 d with fl(d / s) > t (strict) or >= t."""
    def passes(d):
        q = F32(d) / F32(s)
        return q > F32(t) if strict else q >= F32(t)
    T = F32(F32(t) * F32(s))
    up = 0
    while not passes(T):
        T = np.nextafter(T, F32(np.inf))
        up += 1
        assert up < 8
    down = 0
    while T > 0 and passes(np.nextafter(T, F32(0))):
        T = np.nextafter(T, F32(0))
        down += 1
        assert down < 8
    return T


def code_by_thresholds(d: np.ndarray, s: np.float32) -> np.ndarray:
    if s == 0:
        return np.zeros(d.shape, np.int64)
    Ts = [smallest_passing(s, 0.5, True), smallest_passing(s, 1.5, False), smallest_passing(s, 2.5, True)]
    return sum((d >= T).astype(np.int64) for T in Ts)


def _near(x: np.float32, k: int = 3) -> list:
    out = [x]
    lo = hi = x
    for _ in range(k):
        lo = np.nextafter(lo, F32(0))
        hi = np.nextafter(hi, F32(np.inf))
        out += [lo, hi]
    return out


def test_rint_half_even_matches_the_three_comparisons():
    q = np.array([0, 0.25, 0.5, 0.75, 1, 1.25, 1.5, 1.75, 2, 2.5, 2.75, 3, 3.4], F32)
    q = np.concatenate([q, [np.nextafter(F32(v), F32(0)) for v in (0.5, 1.5, 2.5)],
                        [np.nextafter(F32(v), F32(4)) for v in (0.5, 1.5, 2.5)]]).astype(F32)
    by_rint = np.clip(np.rint(q), 0, 3).astype(np.int64)
    by_cmp = (q > F32(0.5)).astype(np.int64) + (q >= F32(1.5)) + (q > F32(2.5))
    assert np.array_equal(by_rint, by_cmp)
    assert by_rint[q == F32(0.5)][0] == 0 and by_rint[q == F32(1.5)][0] == 2 and by_rint[q == F32(2.5)][0] == 2


def test_thresholds_equal_the_division_everywhere():
    rng = np.random.default_rng(20261202)
    scales = np.concatenate([
        F32(10.0) ** rng.uniform(-30, 30, 1500).astype(F32),
        rng.uniform(1e-3, 4, 500).astype(F32),
        np.array([1e-30, 1e30, 1, 1 / 3, 2 / 3, 0.1, 3.0], F32),
    ]).astype(F32)
    checked = 0
    for s in scales:
        s = F32(s)
        d = (rng.uniform(0, 3.2, 600) * s).astype(F32)
        edges = []
        for t in (0.5, 1.5, 2.5):
            edges += _near(F32(F32(t) * s))
            edges += _near(smallest_passing(s, t, t != 1.5))
        d = np.concatenate([d, np.array(edges, F32), np.array([0], F32)]).astype(F32)
        d = d[np.isfinite(d) & (d >= 0)]
        assert np.array_equal(code_by_thresholds(d, s), code_by_division(d, s)), s
        checked += d.size
    assert checked > 1_000_000


def test_zero_scale_gives_code_zero():
    d = np.array([0, 0], F32)
    assert np.array_equal(code_by_thresholds(d, F32(0)), code_by_division(d, F32(0)))
