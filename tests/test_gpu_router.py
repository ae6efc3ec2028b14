"""The router on chosen scores (GPU): exact tiers under heavy ties, ledger reuse across
demote/promote cycles (codes taken back from a freed 2-bit slot, and codes saved to the host
ledger when their slot is handed to another window, then read back), exact bf16 restore on
promotion, pool bookkeeping."""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from oracle.router import EVICTED, FULL, QUANT
from qe_testlib import TIER_CODE, ParityRun

pytestmark = pytest.mark.gpu

WL = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="router", batch=2, n_q_heads=8, n_kv_heads=2,
                         head_dim=128, prefill=32 * 40 + 7, decode_steps=0, window=32, route_period=1, n_sink=5,
                         n_recent=32, kf=8, kq=12, plant_tokens=(), seed=21)


def _scores(event, units, maxw, levels):
    """Seeded scores on a few levels (many exact ties)."""
    k = gen.row_key(WL.seed, gen.T_SCORE, 0, event, np.arange(units)[:, None], np.arange(maxw)[None, :])
    return (gen.splitmix64(k) % np.uint64(levels)).astype(np.float32) / np.float32(4)


@pytest.mark.parametrize("slack", [0, -1], ids=["slack_auto", "no_slack"])
def test_router_cycles_with_ties(slack):
    wl = dataclasses.replace(WL, int2_slack=slack)
    track = [(b, 0, h) for b in range(wl.batch) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, 1, track)
    run.prefill()
    cache = run.cache
    info = cache.layer_info(0)
    units, maxw = info.units, info.max_windows
    kept_before = {}
    n_events = 12
    for event in range(n_events):
        S = _scores(event, units, maxw, levels=3 + event % 6)
        # windows that are evicted keep their (irrelevant) scores; the oracle sees the same floats
        cache.set_scores(0, S)
        for tr in run.tracked:
            u = tr.b * WL.n_kv_heads + tr.kvh
            for j in tr.unit.S:
                tr.unit.S[j] = np.float32(S[u, j])
        cache.qe_route(0)
        tiers = cache.tiers(0)
        for tr in run.tracked:
            res = tr.unit.route()
            u = tr.b * WL.n_kv_heads + tr.kvh
            for j, z in tr.unit.tier.items():
                assert tiers[u, j] == TIER_CODE[z], (event, u, j, tiers[u, j], z)
            run.check_codes(tr)
            run.check_bf16_windows(tr)
    cache.qe_synchronize()
    st = cache.route_stats(0)
    assert st.routes == n_events and st.promotions > 0 and st.ledger_reuses > 0 and st.evictions > 0
    if slack == 0:   # freed slots outlive most returns: codes taken back from their old slot
        assert st.int2_reclaims > 0
    else:            # no spare slot: codes saved to the host ledger before their slot is reused,
        # and read back from it by later re-demotions (their codes were checked above)
        assert st.ledger_writes > 0 and st.ledger_reuses > st.int2_reclaims
    assert run.codes_checked > 0
