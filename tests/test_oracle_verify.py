"""Speculative verify with rollback in the oracle, pinned against the sequential decode steps it
stands for: accepted drafts leave exactly the state of that many decode steps, rejected drafts
leave no trace (H2O page §5: score increments of rejected queries are rolled back)."""
import dataclasses

import numpy as np

import qe_inputs as gen
from oracle.run import make_unit, prefill, step_inputs

WL = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], prefill=255, plant_tokens=())


def _inputs(t0, n):
    qs, ks, vs = [], [], []
    for j in range(n):
        q, k, v = step_inputs(WL, 0, 0, 0, t0 + j)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    return qs, ks, vs


def test_accepted_drafts_equal_sequential_steps():
    for n, acc in ((4, 4), (4, 2), (3, 0), (1, 1)):
        a, b = make_unit(WL), make_unit(WL)
        prefill(WL, a, 0, 0, 0)
        prefill(WL, b, 0, 0, 0)
        qs, ks, vs = _inputs(1, n)
        outs, _ = a.verify(qs, ks, vs)
        seq = [b.decode_step(qs[j], ks[j], vs[j])[0] for j in range(n)]
        for j in range(n):                                 # outputs do not depend on the scores
            assert np.array_equal(outs[j], seq[j])
        a.commit(acc)
        c = make_unit(WL)                                  # the reference: acc decode steps only
        prefill(WL, c, 0, 0, 0)
        for j in range(acc):
            c.decode_step(qs[j], ks[j], vs[j])
        assert a.L == c.L == WL.prefill + acc
        assert a.tier == c.tier
        assert {j: float(x) for j, x in a.S.items()} == {j: float(x) for j, x in c.S.items()}


def test_rejected_draft_closes_the_window_it_opened():
    a = make_unit(WL)
    prefill(WL, a, 0, 0, 0)                                # 255 tokens: the next one opens window 16
    qs, ks, vs = _inputs(1, 3)
    a.verify(qs, ks, vs)
    assert 16 in a.tier
    a.commit(0)
    assert 16 not in a.tier and a.L == 255
    a.verify(qs, ks, vs)
    a.commit(2)
    assert 16 in a.tier and a.L == 257
