"""Routing diagnostics on a running cache: selection churn, cutoff margins, revivals, and the
attention mass the compressed cache has dropped, now and later (future missed mass).

Definitions (QEvict reading notes §3, H2O page §5.1):

* selection churn of a routing event: the Jaccard distance 1 - |A n B| / |A u B| between the
  window sets before (A) and after (B) the event, for the Full set and for the kept set
  (Full or Quantized);
* cutoff margin: the lowest kept score minus the highest dropped score at a cut, here also
  relative to the kept score;
* revivals: Quantized windows promoted back to Full at the event;
* dropped mass at a decode step: the attention mass, under an uncompressed cache, that falls on
  windows the compressed cache has evicted, as a fraction of the step's total (the G query
  heads of a KV head each carry mass 1);
* future missed mass (FMM) of a routing event: the dropped mass of the windows evicted at or
  before that event (eviction is final), averaged over the decode steps that follow it.

The uncompressed distribution comes from a companion cache fed the same inputs whose routing
keeps every window Full (fixed capacities, K_f larger than any window count): its per-window
score increments are the full-attention masses.  Everything here reads the caches through the
C ABI; the numbers are the CUDA path's own.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

from . import TIER_EVICTED, QECache, config_from_workload


def jaccard_distance(both: int, a: int, b: int) -> float:
    union = a + b - both
    return 0.0 if union == 0 else 1.0 - both / union


@dataclasses.dataclass
class EventRecord:
    step: int
    layer: int
    unit: int
    kf: int
    kq: int
    full_churn: float
    kept_churn: float
    full_margin: float        # lowest Full score minus highest non-Full score (inf: no cut)
    kept_margin: float        # lowest kept score minus highest evicted score (inf: no cut)
    full_margin_rel: float
    kept_margin_rel: float
    revivals: int
    demotions: int
    evictions: int


def event_records(cache: QECache, layer: int, step: int) -> List[EventRecord]:
    """Records of the layer's latest routing event, one per unit."""
    out = []
    for u, d in enumerate(cache.route_diag(layer)):
        def margin(kept, nxt):
            if kept < 0 or nxt < 0:
                return float("inf"), float("inf")
            m = float(kept) - float(nxt)
            return m, m / max(float(kept), 1e-30)
        fm, fr = margin(d.full_cut_kept, d.full_cut_next)
        km, kr = margin(d.kept_cut_kept, d.kept_cut_next)
        out.append(EventRecord(step, layer, u, d.kf, d.kq,
                               jaccard_distance(d.full_both, d.full_old, d.full_new),
                               jaccard_distance(d.kept_both, d.kept_old, d.kept_new),
                               fm, km, fr, kr, d.promotions, d.demotions, d.evictions))
    return out


def full_attention_config(wl, max_context: Optional[int] = None, **kw):
    """Configuration of the companion cache: the same shapes, every window kept Full."""
    cfg = config_from_workload(wl, max_context=max_context, **kw)
    cfg.cap_mode = 0
    cfg.kf = (cfg.max_context + cfg.window - 1) // cfg.window + 1
    cfg.kq = 0
    return cfg


class DroppedMass:
    """Per-step dropped mass of every unit of one layer, from the companion cache's score
    increments and the compressed cache's evicted windows."""

    def __init__(self, cache: QECache, full: QECache, layer: int, group: int):
        self.cache, self.full, self.layer, self.G = cache, full, layer, group
        self.prev = full.scores(layer).astype(np.float64)
        self.history: List[np.ndarray] = []        # per step: [units] dropped mass fractions
        self.events: List[tuple] = []              # (step index, evicted mask [units][windows])

    def step(self) -> np.ndarray:
        """Call after each decode step of both caches (before routing); returns the companion's
        per-window mass of the step [units][windows]."""
        cur = self.full.scores(self.layer).astype(np.float64)
        inc = cur - self.prev                      # full-attention mass per window at this step
        self.prev = cur
        evicted = self.cache.tiers(self.layer) == TIER_EVICTED
        self.history.append((inc * evicted).sum(axis=1) / self.G)
        return inc

    def routed(self):
        """Call after a routing event of the compressed cache."""
        self.events.append((len(self.history), self.cache.tiers(self.layer) == TIER_EVICTED))


def run(wl, n_layers: Optional[int] = None, steps: Optional[int] = None, layers_report=(0,), device="cuda:0"):
    """Drive the compressed cache and its companion over the workload (device-side inputs) and
    return per-event records, per-step dropped mass and per-event future missed mass of the
    reported layers."""
    import torch

    import qe_inputs.cuda as gc
    dev = torch.device(device)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    Lyr = n_layers or wl.n_layers
    T = steps or wl.decode_steps
    wl = dataclasses.replace(wl, n_layers=Lyr)
    cache = QECache(config_from_workload(wl), stream.cuda_stream)
    full = QECache(full_attention_config(wl), stream.cuda_stream)
    g = gc.DeviceGenerator(wl, device=dev)
    B, Hkv, Hq, D = wl.batch, wl.n_kv_heads, wl.n_q_heads, wl.head_dim
    kbuf = torch.empty(B, Hkv, wl.prefill, D, device=dev, dtype=torch.int16)
    vbuf = torch.empty_like(kbuf)
    for layer in range(Lyr):
        g.keys_values(layer, 0, wl.prefill, kbuf, vbuf, stream.cuda_stream)
        cache.qe_append(layer, kbuf, vbuf, wl.prefill)
        full.qe_append(layer, kbuf, vbuf, wl.prefill)
    del kbuf, vbuf
    k = torch.empty(B, Hkv, 1, D, device=dev, dtype=torch.int16)
    v = torch.empty_like(k)
    q = torch.empty(B, Hq, D, device=dev, dtype=torch.int16)
    out = torch.empty(B, Hq, D, device=dev, dtype=torch.float32)
    dm = {layer: DroppedMass(cache, full, layer, wl.group) for layer in layers_report}
    incs: Dict[int, List[np.ndarray]] = {layer: [] for layer in layers_report}
    records: List[EventRecord] = []
    for t in range(1, T + 1):
        for layer in range(Lyr):
            g.keys_values(layer, wl.prefill + t - 1, 1, k, v, stream.cuda_stream)
            g.queries(layer, t, q, stream.cuda_stream)
            for c in (cache, full):
                c.qe_append(layer, k, v, 1)
                c.qe_decode_step(layer, q, out)
        for layer in layers_report:
            incs[layer].append(dm[layer].step())
        if t % wl.route_period == 0:
            cache.qe_route(-1)
            full.qe_route(-1)
            for layer in layers_report:
                records.extend(event_records(cache, layer, t))
                dm[layer].routed()
    cache.qe_synchronize()
    full.qe_synchronize()
    fmm = {}
    for layer in layers_report:
        per_event = []
        for idx, evicted in dm[layer].events:
            later = incs[layer][idx:]
            if not later:
                continue
            per_event.append(np.mean([(inc * evicted).sum(axis=1) / wl.group for inc in later], axis=0))
        fmm[layer] = per_event
    dropped = {layer: np.array(dm[layer].history) for layer in layers_report}
    return records, dropped, fmm


def summary(records: List[EventRecord], dropped: Dict[int, np.ndarray], fmm: Dict[int, list]) -> dict:
    """Means and percentiles of the diagnostics over units and events."""
    fin = lambda xs: [x for x in xs if np.isfinite(x)]
    s = {
        "events": len({(r.step, r.layer) for r in records}),
        "full_churn_mean": float(np.mean([r.full_churn for r in records])) if records else 0.0,
        "kept_churn_mean": float(np.mean([r.kept_churn for r in records])) if records else 0.0,
        "revivals_per_event_unit": float(np.mean([r.revivals for r in records])) if records else 0.0,
        "full_margin_rel_p5": float(np.percentile(fin([r.full_margin_rel for r in records]), 5)) if fin(
            [r.full_margin_rel for r in records]) else None,
        "kept_margin_rel_p5": float(np.percentile(fin([r.kept_margin_rel for r in records]), 5)) if fin(
            [r.kept_margin_rel for r in records]) else None,
    }
    for layer, d in dropped.items():
        s[f"layer{layer}_dropped_mass_mean"] = float(d.mean()) if d.size else 0.0
        s[f"layer{layer}_dropped_mass_p99"] = float(np.percentile(d, 99)) if d.size else 0.0
        if fmm.get(layer):
            s[f"layer{layer}_fmm_mean"] = float(np.mean([e.mean() for e in fmm[layer]]))
    if dropped:
        alld = np.concatenate([d.ravel() for d in dropped.values() if d.size]) if any(
            d.size for d in dropped.values()) else np.zeros(0)
        s["dropped_mass_mean"] = float(alld.mean()) if alld.size else 0.0
        s["dropped_mass_p50"] = float(np.percentile(alld, 50)) if alld.size else 0.0
        s["dropped_mass_p99"] = float(np.percentile(alld, 99)) if alld.size else 0.0
        f_all = [e.mean() for l in fmm for e in fmm[l]]
        s["fmm_mean"] = float(np.mean(f_all)) if f_all else 0.0
    return s


if __name__ == "__main__":
    import argparse
    import json
    import qe_inputs as gen
    ap = argparse.ArgumentParser(description="routing diagnostics of a workload on the CUDA path")
    ap.add_argument("--workload", default="llama8b_stack")
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--steps", type=int, default=0)
    a = ap.parse_args()
    wl = gen.WORKLOADS[a.workload]
    rec, dropped, fmm = run(wl, n_layers=a.layers or None, steps=a.steps or None,
                            layers_report=tuple(range(a.layers or wl.n_layers)))
    full = summary(rec, dropped, fmm)
    print(json.dumps({"workload": a.workload, **{k: v for k, v in full.items() if not k.startswith("layer")}}))
