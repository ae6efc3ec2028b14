"""Pins of the five-tier per-token oracle (HqeKV reading notes) against what the pages and the
mathematics fix: the section 3.7 worked example, normal quantiles, the eq. (4) decision written
out literally, exact fma rounding, eq. (2) bounds, full attention when nothing is compressed,
mass conservation, the scoring window and demote-only re-ranking."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import hqekv as H

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_worked_example_ranks_into_the_printed_tiers():
    g = json.load(open(os.path.join(GOLD, "hqekv_toy_chunk.json")))
    A, R = np.array(g["attention"]), np.array(g["value_range"])
    joint = H.joint_metric(A, R)
    assert np.allclose(np.round(joint, 3), g["joint_metric_printed"], atol=1e-12)
    names = g["tokens"]
    order = [names[i] for i in np.lexsort((np.arange(8), -joint))]
    assert order == g["order_printed"]
    tiers = H.rank_tiers(joint, np.arange(8), (0, 2, 2, 2))
    got = {k: [names[i] for i in np.flatnonzero(tiers == z)] for k, z in
           (("int4", H.INT4), ("int2", H.INT2), ("nq1", H.NQ1), ("evicted", H.EVICT))}
    for k, v in g["tiers_printed"].items():
        assert sorted(got[k]) == sorted(v), k
    # the notes' remark: attention alone evicts t6 and keeps t7
    t_att = H.rank_tiers(A, np.arange(8), (0, 2, 2, 2))
    assert t_att[5] == H.EVICT and t_att[6] != H.EVICT


def test_rank_ties_go_to_the_lower_position():
    imp = np.array([1.0, 2.0, 2.0, 1.0, 0.0, 2.0], np.float32)
    tiers = H.rank_tiers(imp, np.arange(6), (1, 1, 1, 1))
    # order: 1, 2, 5 (score 2, by position), then 0, 3 (score 1), then 4
    assert tiers.tolist() == [H.NQ1, H.BF16, H.INT4, H.EVICT, H.EVICT, H.INT2]


def test_normal_centers_are_standard_normal_quantiles():
    from scipy.special import ndtr, ndtri      # an independent implementation
    for b in (1, 2, 3):
        c = H.normal_centers(b)
        p = (np.arange(1 << b) + 0.5) / (1 << b)
        assert np.array_equal(c.astype(np.float32), ndtri(p).astype(np.float32)), b
        assert np.max(np.abs(ndtr(c) - p)) < 1e-15
        beta = H.normal_boundaries(b)
        assert np.max(np.abs(ndtr(beta) - (np.arange(1, 1 << b) / (1 << b)))) < 1e-15
    assert H.normal_boundaries(1).tolist() == [0.0]
    assert abs(H.normal_centers(1)[1] - 0.6745) < 5e-5 and H.normal_centers(1)[0] == -H.normal_centers(1)[1]


def test_normal_decision_is_the_literal_eq4_argmin():
    from scipy.special import ndtr
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((200, 64)) * rng.uniform(0.1, 5, (200, 1)) + rng.normal(0, 2, (200, 1))).astype(np.float32)
    for b in (1, 2, 3):
        codes, m, s = H.normal_quantize(x, b)
        xp = (x.astype(np.float64) - m.astype(np.float64)[:, None]) / s.astype(np.float64)[:, None]
        c = H.normal_centers(b)
        dist = np.abs(ndtr(c)[None, None, :] - ndtr(xp)[:, :, None])     # eq. (4): mass between
        lit = np.argmin(dist, axis=2)                                    # first (lower) on ties
        near = np.min(np.abs(xp[:, :, None] - H.normal_boundaries(b)[None, None, :]), axis=2) < 1e-9 if b > 1 else \
            np.abs(xp) < 1e-9
        assert np.array_equal(codes[~near], lit[~near].astype(np.uint8)), b


def test_one_bit_code_is_the_sign_against_the_mean():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((100, 128)).astype(np.float32)
    x[0] = np.where(np.arange(128) % 2 == 0, 1.0, -1.0)      # mean exactly 0: half the values tie
    x[1] = 0.5                                               # constant: s = 0, codes 0
    codes, m, s = H.normal_quantize(x, 1)
    assert m[0] == 0 and np.array_equal(codes[0], (x[0] > 0).astype(np.uint8))
    assert s[1] == 0 and not codes[1].any()
    assert np.array_equal(codes[2:], (x[2:] > m[2:, None]).astype(np.uint8))


def test_mean_std_match_the_closed_form():
    rng = np.random.default_rng(5)
    for D in (64, 128):
        x = (rng.standard_normal((50, D)) * 3 + 1).astype(np.float32)
        m, s = H.mean_std_f32(x)
        xd = x.astype(np.float64)
        assert m.dtype == np.float32 and s.dtype == np.float32
        assert np.allclose(m, xd.mean(axis=1), rtol=1e-6, atol=1e-6)
        assert np.allclose(s, xd.std(axis=1), rtol=1e-6)


def _f32_neighbours(c):
    c = np.float32(c)
    out = {float(c)}
    lo = hi = c
    for _ in range(3):
        lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(hi, np.float32(np.inf))
        out |= {float(lo), float(hi)}
    return sorted(v for v in out if math.isfinite(v))


def _even(v):
    return int(np.array([v], np.float32).view(np.uint32)[0]) & 1 == 0


def _nearest_f32(t: Fraction) -> float:
    """The float32 nearest the rational t (ties to even), by exact comparison among the float32
    values around float(t)."""
    best = None
    for c in _f32_neighbours(float(t)):
        d = abs(Fraction(c) - t)
        if best is None or d < best[0] or (d == best[0] and _even(c)):
            best = (d, c)
    return best[1]


def _nearest_f32_sqrt(v: Fraction) -> float:
    """The float32 nearest sqrt(v) (ties to even): candidate c_i wins when sqrt(v) lies between
    the midpoints it shares with its neighbours, decided by comparing v with their squares."""
    cands = [c for c in _f32_neighbours(math.sqrt(float(v))) if c >= 0]
    for i, c in enumerate(cands):
        lo = (Fraction(cands[i - 1]) + Fraction(c)) / 2 if i > 0 else None
        hi = (Fraction(c) + Fraction(cands[i + 1])) / 2 if i + 1 < len(cands) else None
        above_lo = lo is None or v > lo * lo or (v == lo * lo and _even(c))
        below_hi = hi is None or v < hi * hi or (v == hi * hi and _even(c))
        if above_lo and below_hi:
            return c
    raise AssertionError("sqrt outside the candidates")


def _adversarial_rows(D, rng):
    rows = []
    big = np.float32(3e38)
    rows.append(np.full(D, big, np.float32))                        # a float32 sum would overflow
    r = np.ones(D, np.float32); r[-1] = np.float32(1 + 2.0 ** -17)  # mean exactly between 1 and
    rows.append(r)                                                  # its successor: ties to even
    r = np.zeros(D, np.float32); r[3] = np.float32(1.5)             # one nonzero value
    rows.append(r)
    r = (rng.standard_normal(D) * 1e3).astype(np.float32)           # cancellation: +-x pairs and a
    r[D // 2:] = -r[:D // 2]; r[0] = np.float32(r[0] + np.float32(1e-3))   # small residual
    rows.append(r)
    r = rng.standard_normal(D).astype(np.float32)                   # magnitudes 2^-100 .. 2^100
    r *= np.exp2(rng.integers(-100, 101, D)).astype(np.float32)
    rows.append(r)
    r = (rng.integers(1, 1000, D) * 2.0 ** -149).astype(np.float32)  # subnormals only
    rows.append(r)
    r = rng.standard_normal(D).astype(np.float32); r[::7] = np.float32(1e-30)   # tiny beside O(1)
    rows.append(r)
    rows.append(np.full(D, np.float32(-2.75), np.float32))           # constant row: s = 0
    r = rng.standard_normal(D).astype(np.float32); r[5] = np.float32(1e30)      # one huge value
    rows.append(r)
    return np.stack(rows)


def test_mean_std_are_the_exact_values_rounded_once():
    """eq. (3)'s mean and population std: the exact values for the row, rounded once to the
    nearest float32 (ties to even), against Fraction arithmetic, bit for bit, on random rows and
    on rows chosen to break any fixed-order float32 or float64 summation."""
    rng = np.random.default_rng(31)
    for D in (64, 128):
        x = np.concatenate([(rng.standard_normal((12, D)) * rng.uniform(0.1, 10, (12, 1))).astype(np.float32),
                            _adversarial_rows(D, rng)])
        m, s = H.mean_std_f32(x)
        for r in range(x.shape[0]):
            fx = [Fraction(float(v)) for v in x[r]]
            mu = sum(fx) / D
            var = sum((f - mu) ** 2 for f in fx) / D
            assert float(m[r]) == _nearest_f32(mu), (D, r, m[r], float(mu))
            assert float(s[r]) == _nearest_f32_sqrt(var), (D, r, s[r], math.sqrt(float(var)))
    # the tie row: exact mean 1 + 2^-24 lies halfway between 1 and 1 + 2^-23, so it rounds to 1
    m, _ = H.mean_std_f32(_adversarial_rows(128, rng)[1:2])
    assert m[0] == np.float32(1.0)
    # the row whose float32 sum would overflow still has mean 3e38 and std 0
    m, s = H.mean_std_f32(_adversarial_rows(64, rng)[0:1])
    assert m[0] == np.float32(3e38) and s[0] == 0


def test_mean_std_closed_forms_of_structured_rows():
    # one nonzero value a among D: mean a / D (exact, D a power of two), std |a| sqrt(D - 1) / D
    for D in (64, 128):
        for a in (1.5, -3.0, 1e-20, 7e30):
            x = np.zeros((1, D), np.float32)
            x[0, 0] = np.float32(a)
            m, s = H.mean_std_f32(x)
            assert m[0] == np.float32(np.float32(a) / D)
            want = _nearest_f32_sqrt(Fraction(float(np.float32(a))) ** 2 * (D - 1) / D ** 2)
            assert float(s[0]) == want
    # two values +-c in equal numbers: mean 0, std |c| exactly
    x = np.tile(np.array([2.5, -2.5], np.float32), 64)[None, :]
    m, s = H.mean_std_f32(x)
    assert m[0] == 0 and s[0] == np.float32(2.5)


def test_fmaf32_rounds_once():
    rng = np.random.default_rng(6)
    a = rng.standard_normal(3000).astype(np.float32)
    b = rng.standard_normal(3000).astype(np.float32)
    c = (rng.standard_normal(3000) * 64).astype(np.float32)
    r = H.fmaf32(a, b, c)

    def exact(a, b, c):
        x = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
        f = np.float32(float(x))
        cand = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
        return min(cand, key=lambda y: (abs(Fraction(float(y)) - x), int(np.float32(y).view(np.uint32)) & 1))
    assert all(exact(a[i], b[i], c[i]) == r[i] for i in range(3000))
    # a double rounding trap: the float64 sum lands on a float32 midpoint the exact sum is below
    a1 = np.float32(2.0 ** -24 * (1 + 2.0 ** -15))
    b1 = np.float32(1 - 2.0 ** -15)
    c1 = np.float32(1 + 2.0 ** -23)
    naive = np.float32(np.float64(a1) * np.float64(b1) + np.float64(c1))
    assert naive == np.float32(1 + 2.0 ** -22)
    assert H.fmaf32(a1, b1, c1) == c1 == exact(a1, b1, c1)


def test_uniform_token_quantizer_bounds():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 128)) * rng.uniform(0.01, 10, (64, 1))).astype(np.float32)
    for bits in (4, 2):
        codes, z, s = H.uniform_quantize_rows(x, bits)
        assert codes.max() <= (1 << bits) - 1
        xh = H.uniform_dequantize_rows(codes, z, s)
        assert np.all(np.abs(x - xh) <= s[:, None] / 2 * (1 + 1e-5) + 1e-6 * np.abs(x))
        amin = np.argmin(x, axis=1)
        assert np.array_equal(xh[np.arange(64), amin], z)


def test_tier_counts_of_the_16k_workload():
    # 10 / 20 / 30 / 30 % of L, BF16 share including 5 sink + 32 recent tokens, the rest evicted
    assert H.tier_counts(16448, 5, 32, (0.10, 0.20, 0.30, 0.30)) == (1607, 3289, 4934, 4934)
    assert H.tier_counts(100, 5, 32, (0.10, 0.20, 0.30, 0.30)) == (0, 20, 30, 30)


def _unit(**kw):
    args = dict(head_dim=32, group=2, n_sink=2, n_recent=4, period=8, score_window=3,
                fractions=(0.2, 0.2, 0.2, 0.2), max_context=200)
    args.update(kw)
    return H.HqeUnit(**args)


def _bf16(x):
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32)


def test_uncompressed_unit_is_full_attention():
    rng = np.random.default_rng(8)
    u = _unit(fractions=(1.0, 0.0, 0.0, 0.0))
    K = _bf16(rng.standard_normal((60, 32)))
    V = _bf16(rng.standard_normal((60, 32)))
    u.append(K[:40], V[:40])
    for t in range(20):
        q = _bf16(rng.standard_normal((2, 32)))
        o, mass = u.decode_step(q, K[40 + t], V[40 + t])
        n = 41 + t
        lg = q.astype(np.float64) @ K[:n].T.astype(np.float64) / math.sqrt(32)
        p = np.exp(lg - lg.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        assert np.allclose(o, p @ V[:n].astype(np.float64), rtol=1e-12, atol=1e-13)
        assert abs(sum(mass.values()) + p[:, :2].sum() - 2.0) < 1e-12      # mass conservation
    assert u.tier_histogram()[0] == 60


def test_rerank_demotes_only_and_fills_the_fractions_first():
    rng = np.random.default_rng(9)
    u = _unit()
    u.append(_bf16(rng.standard_normal((120, 32))), _bf16(rng.standard_normal((120, 32))))
    prev = u.tier[:u.L].copy()
    for t in range(1, 41):
        q = _bf16(rng.standard_normal((2, 32)) * 2)
        k, v = _bf16(rng.standard_normal((1, 32))), _bf16(rng.standard_normal((1, 32)))
        S_before = u.S.copy()
        u.decode_step(q, k, v)
        if not u.scoring_step(t):
            assert np.array_equal(u.S, S_before)
        if t % 8 == 0:
            res = u.history[-1]
            assert not u.S.any()                                   # rolling window restarts
            assert np.all(u.tier[:len(prev)] >= prev)              # demote only
            if t == 8:                                              # everything was BF16: counts exact
                cnt = np.bincount([z for z in res.desired.values()], minlength=5)
                assert tuple(cnt[:4]) == res.counts
                hist = u.tier_histogram()
                assert hist[1:4] == res.counts[1:]
            for p, (z0, zn) in res.changed.items():
                assert zn > z0
            prev = u.tier[:u.L].copy()
        assert np.all(u.tier[:2] == H.BF16) and np.all(u.tier[u.L - 4:u.L] == H.BF16)


def test_requantization_starts_from_the_current_codes():
    rng = np.random.default_rng(10)
    k = _bf16(rng.standard_normal(64) * 3)
    v = _bf16(rng.standard_normal(64))
    q4 = H.quantize_token(H.INT4, k, v)
    k4, v4 = H.dequantize_token(q4)
    via = H.quantize_token(H.INT2, k4, v4)
    direct = H.quantize_token(H.INT2, k, v)
    # the chain keeps min and max of the 4-bit reconstruction: min exactly, codes mostly agree
    assert via.k_p0 == q4.k_p0 and np.mean(via.k_codes == direct.k_codes) > 0.8
    k1, _ = H.dequantize_token(H.quantize_token(H.NQ1, k4, v4))
    m, s = H.mean_std_f32(k4[None, :])
    assert set(np.round((k1.astype(np.float64) - m[0]) / s[0], 4)) <= {-0.6745, 0.6745}
