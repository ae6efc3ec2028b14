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


def test_mean_std_exact_when_every_step_is_exact():
    # integer rows with a sum divisible by D: every add, the division by D, x - m and (x - m)^2
    # are exact in float32, so m and the variance are exact and s is the rounded square root
    rng = np.random.default_rng(11)
    for D in (64, 128):
        x = rng.integers(-100, 101, (40, D)).astype(np.int64)
        x[:, -1] -= x.sum(axis=1) % D          # sum divisible by D (the last value moves a little)
        m, s = H.mean_std_f32(x.astype(np.float32))
        me = x.sum(axis=1) // D
        var = ((x - me[:, None]) ** 2).sum(axis=1) / D
        assert np.array_equal(m, me.astype(np.float32))
        assert np.array_equal(s, np.sqrt(var).astype(np.float32))


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
