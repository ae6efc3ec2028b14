"""Drive one cache unit of a workload through prefill and decode steps.

Test infrastructure (see ``oracle/__init__``).

QEvict reading notes, §2 Figure 1 (all windows start in full precision) and
§4.2 (a routing event every Omega generated tokens): the prefill appends L0
tokens with no attention and zero scores; decode step t (1-based) appends
position L0 + t - 1, attends, accumulates, and routes when t % Omega == 0.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional

import numpy as np

import qe_inputs as gen

from .budget import capacities
from .hqekv import HqeUnit
from .qevict import QEvictUnit
from .router import RouteResult


def make_unit(wl, max_context: Optional[int] = None):
    """A QEvict unit, or a five-tier per-token unit for workloads with tiering "tokens"."""
    if wl.tiering == "tokens":
        return HqeUnit(wl.head_dim, wl.group, wl.n_sink, wl.n_recent, wl.route_period, wl.score_window,
                       (wl.frac_bf16, wl.frac_int4, wl.frac_int2, wl.frac_nq1), max_context or wl.max_context)
    return QEvictUnit(wl.window, wl.n_sink, wl.n_recent, wl.head_dim, wl.group,
                      lambda L: capacities(wl, L), max_context or wl.max_context,
                      rope_base=getattr(wl, "rope_theta", 0.0))


def prefill(wl, unit: QEvictUnit, b: int, layer: int, kvh: int, n: Optional[int] = None):
    n = wl.prefill if n is None else n
    kb, vb = gen.gen_keys_values(wl, b, layer, kvh, 0, n)
    unit.append(gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb))


def step_inputs(wl, b: int, layer: int, kvh: int, t: int):
    """(q [G, d], k [1, d], v [1, d]) as float32 bf16 values for decode step t."""
    heads = range(kvh * wl.group, (kvh + 1) * wl.group)
    q = gen.bf16_bits_to_f32(gen.gen_queries(wl, b, layer, heads, t))
    kb, vb = gen.gen_keys_values(wl, b, layer, kvh, wl.prefill + t - 1, 1)
    return q, gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb)


@dataclasses.dataclass
class UnitRun:
    unit: QEvictUnit
    outputs: List[np.ndarray]           # per step, o [G, d] float64
    masses: List[dict]
    sink_mass: List[float]
    routes: List[RouteResult]


def run_unit(wl, b: int, layer: int, kvh: int, n_steps: int,
             on_step: Optional[Callable[[int, QEvictUnit], None]] = None) -> UnitRun:
    unit = make_unit(wl)
    prefill(wl, unit, b, layer, kvh)
    outs, masses, sinks, routes = [], [], [], []
    for t in range(1, n_steps + 1):
        q, k, v = step_inputs(wl, b, layer, kvh, t)
        o, m, s = unit.decode_step(q, k, v)
        outs.append(o)
        masses.append(m)
        sinks.append(s)
        if t % wl.route_period == 0:
            routes.append(unit.route())
        if on_step is not None:
            on_step(t, unit)
    return UnitRun(unit, outs, masses, sinks, routes)
