"""Host arithmetic of the routing diagnostics (no GPU)."""
import numpy as np
import pytest

from tiered_quantize_evict_gb300.diagnostics import EventRecord, jaccard_distance, summary


def test_jaccard_distance():
    assert jaccard_distance(3, 3, 3) == 0.0            # same set
    assert jaccard_distance(0, 2, 2) == 1.0            # disjoint sets
    assert jaccard_distance(1, 2, 2) == pytest.approx(1 - 1 / 3)
    assert jaccard_distance(0, 0, 0) == 0.0            # both empty: no change


def test_summary_means_and_percentiles():
    recs = [EventRecord(16, 0, u, 2, 12, 0.5 * u, 0.25, 1.0, float("inf"), 0.1 * (u + 1), float("inf"), u, 0, 1)
            for u in range(4)]
    dropped = {0: np.array([[0.0, 0.1, 0.2, 0.3]])}
    s = summary(recs, dropped, {0: [np.array([0.2, 0.4])]})
    assert s["events"] == 1
    assert s["full_churn_mean"] == pytest.approx(0.75)
    assert s["kept_churn_mean"] == pytest.approx(0.25)
    assert s["revivals_per_event_unit"] == pytest.approx(1.5)
    assert s["kept_margin_rel_p5"] is None              # no finite kept margin
    assert s["layer0_dropped_mass_mean"] == pytest.approx(0.15)
    assert s["layer0_fmm_mean"] == pytest.approx(0.3)
