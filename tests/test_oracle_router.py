"""Pins of the oracle's routing (no GPU).

The tier of a candidate is fixed by its rank alone; the tests recompute that
rank by counting (how many candidates beat it: higher score, or equal score
and lower window index) instead of sorting, and check the state machine's
invariants over whole trajectories: capacities respected, Evicted final,
the ledger's codes identical on every re-demotion, pinned windows never
ranked.  The H2O page's four scenario families (§5.1) drive the router
with injected masses.
"""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from oracle.qevict import QEvictUnit
from oracle.router import EVICTED, FULL, PINNED, QUANT, assign, candidate_pool
from oracle.run import run_unit

RNG = np.random.default_rng(5)


@pytest.mark.parametrize("n,kf,kq", [(1, 0, 0), (7, 3, 4), (50, 5, 20), (300, 80, 256), (40, 0, 10), (40, 50, 0)])
def test_assignment_equals_counting_rank(n, kf, kq):
    for trial in range(20):
        cands = sorted(RNG.choice(1000, n, replace=False).tolist())
        vals = RNG.integers(0, 4, n).astype(np.float32) / np.float32(3)      # many ties
        scores = {j: np.float32(v) for j, v in zip(cands, vals)}
        res = assign(cands, scores, kf, kq)
        for j in cands:
            r = sum(1 for i in cands if scores[i] > scores[j] or (scores[i] == scores[j] and i < j))
            want = FULL if r < kf else QUANT if r < kf + kq else EVICTED
            got = FULL if j in res.full else QUANT if j in res.quant else EVICTED
            assert got == want
        assert len(res.full) == min(kf, n) and len(res.quant) == min(kq, max(0, n - kf))


def test_candidate_pool_excludes_recent_and_evicted():
    tier = {0: FULL, 1: QUANT, 2: EVICTED, 3: PINNED, 4: PINNED, 5: PINNED}
    # L = 96, w = 16, recent 32 -> aged iff (j+1)*16 <= 64 -> j <= 3
    assert candidate_pool(tier, 96, 16, 32) == [0, 1, 3]


def _trajectory_invariants(wl, b=0, layer=0, kvh=0, steps=None):
    first_pack = {}
    seen_evicted = set()
    prev = {}

    def cb(t, u):
        nonlocal prev
        for j, z in u.tier.items():
            if j in seen_evicted:
                assert z == EVICTED
            if z == EVICTED:
                seen_evicted.add(j)
            if z == QUANT:
                e = u.ledger[j]
                if j in first_pack:
                    assert first_pack[j].equal(e)
                else:
                    first_pack[j] = e
        if t % wl.route_period == 0:
            res = u.history[-1]
            assert len(res.full) <= res.kf and len(res.quant) <= res.kq
            for j, z in u.tier.items():
                lo, hi = u.window_range(j)
                if z == PINNED:
                    assert (j + 1) * wl.window > u.L - wl.n_recent or hi - lo < wl.window - (wl.n_sink if j == 0 else 0)
                if z in (FULL, QUANT):
                    assert (j + 1) * wl.window <= u.L - wl.n_recent
        prev = dict(u.tier)

    return run_unit(wl, b, layer, kvh, steps or wl.decode_steps, cb), first_pack


def test_tiny_workload_invariants_and_planted_window():
    wl = gen.WORKLOADS["tiny_qevict"]
    run, packs = _trajectory_invariants(wl)
    hist = [(r, dict()) for r in run.routes]
    # the planted window 4 (tokens 64..79) is demoted to INT2 before the queries carry the
    # planted direction (step 40) and promoted back to BF16 afterwards
    tiers = []
    for i, r in enumerate(run.routes):
        t = (i + 1) * wl.route_period
        z = FULL if 4 in r.full else QUANT if 4 in r.quant else EVICTED
        tiers.append((t, z))
    before = [z for t, z in tiers if t < wl.plant_step]
    after = [z for t, z in tiers if t > wl.plant_step]
    assert QUANT in before and EVICTED not in before
    assert after[-1] == FULL
    # its ledger entry was made once and is unchanged
    assert 4 in packs
    # mass conservation every step: window masses + sink mass = G
    for m, s in zip(run.masses, run.sink_mass):
        assert abs(sum(m.values()) + s - wl.group) < 1e-9


def _unit(kf, kq, w=8, n_sink=0, n_recent=8):
    return QEvictUnit(w, n_sink, n_recent, 16, 1, lambda L: (kf, kq), 4096)


def _drive(u, mass_fn, steps, omega, L0=128):
    u.append(np.zeros((L0, 16), np.float32), np.zeros((L0, 16), np.float32))
    hist = []
    for t in range(1, steps + 1):
        u.append(np.zeros((1, 16), np.float32), np.zeros((1, 16), np.float32))
        live = [j for j, z in u.tier.items() if z != EVICTED]
        u.accumulate({j: mass_fn(t, j) for j in live})
        if t % omega == 0:
            hist.append(u.route())
    return hist


def test_scenario_uniform_has_age_bias():
    """Uniform attention: older windows have accumulated as much per step; ties go to lower positions."""
    u = _unit(kf=3, kq=2)
    hist = _drive(u, lambda t, j: 0.01, 16, 8)
    assert hist[0].full == [0, 1, 2] and hist[0].quant == [3, 4]


def test_scenario_distant_hotspot_is_kept():
    u = _unit(kf=2, kq=2)
    hist = _drive(u, lambda t, j: 1.0 if j == 1 else 0.01 * (j % 3), 64, 8)
    assert all(1 in h.full for h in hist)


def test_scenario_hotspot_switch_leaves_residual():
    """Window 2 is hot first, then window 9: 2 keeps its slot on its history alone, 9 rises to Full."""
    def mass(t, j):
        if j == 2:
            return 1.0 if t <= 32 else 0.0
        if j == 9:
            return 0.5 if t <= 32 else 1.0
        return 0.01 * (j % 3)
    u = _unit(kf=2, kq=2)
    hist = _drive(u, mass, 96, 8)
    assert hist[3].full == [2, 9]            # t = 32
    assert 2 in hist[-1].full and 9 in hist[-1].full and hist[-1].order[0] == 9


def test_scenario_delayed_first_reference_is_recoverable_only_with_int2():
    """Window 5 gets no attention until step 40, then all of it.

    With K_q = 0 (H2O's binary eviction) it is gone for good; with an INT2 tier it survives
    as Quantized and is promoted once its score overtakes (QEvict notes, eq. (6))."""
    def mass(t, j):
        if t <= 40:
            return 0.0 if j == 5 else 0.05 * ((j * 7) % 5 + 1)
        return 3.0 if j == 5 else 0.05 * ((j * 7) % 5 + 1)
    u = _unit(kf=2, kq=0)
    hist = _drive(u, mass, 96, 8)
    assert 5 in hist[0].evicted and u.tier[5] == EVICTED
    u = _unit(kf=2, kq=24)
    hist = _drive(u, mass, 96, 8)
    assert 5 in hist[0].quant and 5 in hist[-1].full
