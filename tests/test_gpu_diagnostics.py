"""Routing diagnostics of the CUDA path against the oracle (GPU).

The Llama-shaped byte-budget stack (2 layers, 64 decode steps, routing every 16) runs on the
compressed cache and on a companion cache that keeps every window Full.  For every unit of both
layers the oracle runs the same pair of units.  Compared:

- each routing event's record: set sizes and overlaps, moves, and the scores at both cuts;
- selection churn of the Full and kept sets, recomputed here from the oracle's sets;
- the per-step dropped mass: full-attention mass on the compressed cache's evicted windows;
- the future missed mass of each routing event, recomputed here from the oracle's full-attention
  masses and the windows evicted by then.

A unit whose record differs from the oracle's at a tie-ambiguous cut (margin below 1e-4
relative) would stop being compared, as in the trajectory tests; the test fails if that happens.
"""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from oracle.qevict import QEvictUnit
from oracle.router import EVICTED, FULL, QUANT
from oracle.run import make_unit, prefill, step_inputs

pytestmark = pytest.mark.gpu

SCORE_RTOL = 1e-4
MARGIN_RTOL = 1e-4
MASS_ATOL = 1e-4


def _full_unit(wl):
    return QEvictUnit(wl.window, wl.n_sink, wl.n_recent, wl.head_dim, wl.group,
                      lambda L: (10 ** 6, 0), wl.max_context)


def test_diagnostics_match_oracle():
    from tiered_quantize_evict_gb300 import diagnostics as dg
    wl = dataclasses.replace(gen.WORKLOADS["llama8b_stack"], n_layers=2)
    T = 64
    records, dropped, fmm = dg.run(wl, steps=T, layers_report=(0, 1))
    rec = {(r.step, r.layer, r.unit): r for r in records}
    checked_events = checked_steps = checked_fmm = 0
    ambiguous = []
    for layer in (0, 1):
        for kvh in range(wl.n_kv_heads):
            u, f = make_unit(wl), _full_unit(wl)
            prefill(wl, u, 0, layer, kvh)
            prefill(wl, f, 0, layer, kvh)
            live = True
            full_mass = []        # full-attention window masses of every step
            evicted_at = []       # (steps done, windows evicted by then) after each routing event
            for t in range(1, T + 1):
                q, k, v = step_inputs(wl, 0, layer, kvh, t)
                u.decode_step(q, k, v)
                _, mass_full, _ = f.decode_step(q, k, v)
                full_mass.append(mass_full)
                if live:
                    ref = sum(m for j, m in mass_full.items() if u.tier.get(j) == EVICTED) / wl.group
                    got = dropped[layer][t - 1][kvh]
                    assert abs(got - ref) <= MASS_ATOL, (layer, kvh, t, got, ref)
                    checked_steps += 1
                if t % wl.route_period:
                    continue
                old = dict(u.tier)
                res = u.route()
                f.route()
                evicted_at.append((t, {j for j, z in u.tier.items() if z == EVICTED}))
                if not live:
                    continue
                r = rec[(t, layer, kvh)]
                amb = min(res.margin_f / max(float(u.S[res.order[res.kf - 1]]), 1e-30) if 0 < res.kf < len(res.order) else 1.0,
                          res.margin_q / max(float(u.S[res.order[res.kf + res.kq - 1]]), 1e-30)
                          if 0 < res.kf + res.kq < len(res.order) else 1.0)
                new = u.tier
                fo = {j for j, z in old.items() if z == FULL}
                fn = {j for j, z in new.items() if z == FULL}
                ko = fo | {j for j, z in old.items() if z == QUANT}
                kn = fn | {j for j, z in new.items() if z == QUANT}
                want = dict(kf=res.kf, kq=res.kq, full_old=len(fo), full_new=len(fn), full_both=len(fo & fn),
                            kept_old=len(ko), kept_new=len(kn), kept_both=len(ko & kn),
                            promotions=len([j for j in res.full if old[j] == QUANT]),
                            demotions=len([j for j in res.quant if old[j] == FULL]),
                            evictions=len(res.evicted))
                got = dict(kf=r.kf, kq=r.kq, revivals=r.revivals, demotions=r.demotions, evictions=r.evictions)
                same = (r.kf, r.kq, r.revivals, r.demotions, r.evictions) == (
                    want["kf"], want["kq"], want["promotions"], want["demotions"], want["evictions"])
                if not same and amb <= MARGIN_RTOL:
                    live = False   # both outcomes are correct; the runs diverge from here
                    ambiguous.append((layer, kvh, t, amb))
                    continue
                assert same, (t, layer, kvh, got, want)
                # selection churn: Jaccard distance 1 - |A n B| / |A u B| of the sets before and after
                for name, a_set, b_set in (("full_churn", fo, fn), ("kept_churn", ko, kn)):
                    union = len(a_set | b_set)
                    ref = 0.0 if union == 0 else 1.0 - len(a_set & b_set) / union
                    assert getattr(r, name) == pytest.approx(ref, abs=1e-12), (name, t, layer, kvh)
                def cut(rank):
                    return float(u.S[res.order[rank]]) if 0 <= rank < len(res.order) else None
                for name, rank in (("full_margin", res.kf), ("kept_margin", res.kf + res.kq)):
                    a, b = cut(rank - 1), cut(rank)
                    m = getattr(r, name)
                    if a is None or b is None:
                        assert m == float("inf")
                    else:
                        assert m == pytest.approx(a - b, rel=0, abs=SCORE_RTOL * a + 1e-6), (name, t, m, a - b)
                checked_events += 1
            # future missed mass of each event followed by decode steps: the full-attention mass
            # (per query head) on the windows evicted by then, averaged over the later steps
            for e, (t_ev, ev_set) in enumerate(evicted_at):
                later = full_mass[t_ev:]
                if not later or any(a[0] == layer and a[1] == kvh and a[2] <= t_ev for a in ambiguous):
                    continue
                ref = np.mean([sum(m for j, m in fm.items() if j in ev_set) / wl.group for fm in later])
                assert abs(fmm[layer][e][kvh] - ref) <= MASS_ATOL, (layer, kvh, t_ev, fmm[layer][e][kvh], ref)
                checked_fmm += 1
    assert not ambiguous, f"units no longer compared: {ambiguous}"
    assert checked_events > 0 and checked_steps > 0 and checked_fmm > 0
    s = dg.summary(records, dropped, fmm)
    print(f"diagnostics parity: {checked_events} unit events, {checked_steps} unit steps, {checked_fmm} FMM values; "
          f"summary {s}")
