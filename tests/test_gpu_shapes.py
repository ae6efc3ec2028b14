"""Trajectory parity over a sweep of shapes and capacity rules (GPU).

Small enough for the oracle to follow every unit through every step; each case spans
several tiles per warp, ragged lengths (prefill not a multiple of w) and several routing
events."""
import dataclasses

import pytest

import qe_inputs as gen
from qe_testlib import ParityRun

pytestmark = pytest.mark.gpu

BASE = gen.WORKLOADS["tiny_qevict"]

CASES = {
    # d=128, w=32, G=4, 4 units, ragged prefill
    "d128_w32_g4": dataclasses.replace(BASE, name="d128_w32_g4", batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128,
                                       prefill=300, decode_steps=40, window=32, route_period=8, n_sink=5,
                                       n_recent=32, kf=4, kq=6, plant_tokens=(), seed=11),
    # d=64, w=64, G=2, no sink
    "d64_w64_g2": dataclasses.replace(BASE, name="d64_w64_g2", batch=1, n_q_heads=6, n_kv_heads=3, head_dim=64,
                                      prefill=520, decode_steps=36, window=64, route_period=12, n_sink=0,
                                      n_recent=20, kf=2, kq=3, plant_tokens=(), seed=12),
    # d=128, w=16, G=1, long sink, one recent token
    "d128_w16_g1": dataclasses.replace(BASE, name="d128_w16_g1", batch=3, n_q_heads=1, n_kv_heads=1, head_dim=128,
                                       prefill=100, decode_steps=30, window=16, route_period=5, n_sink=15,
                                       n_recent=1, kf=3, kq=2, plant_tokens=(), seed=13),
    # token-share capacities (cap_mode 1), 2 layers
    "shares_2layers": dataclasses.replace(gen.WORKLOADS["throughput_32k"], name="shares_2layers", batch=2,
                                          n_layers=2, prefill=640, decode_steps=48, route_period=16,
                                          frac_bf16=0.3, frac_int2=0.3, seed=14),
    # byte-budget capacities (cap_mode 2), the Llama-shaped stack cut to 2 layers
    "budget_2layers": dataclasses.replace(gen.WORKLOADS["llama8b_stack"], name="budget_2layers", n_layers=2,
                                          decode_steps=64),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_trajectory_parity(name):
    wl = CASES[name]
    track = [(b, l, h) for b in range(wl.batch) for l in range(wl.n_layers) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, wl.n_layers, track)
    run.prefill()
    for _ in range(wl.decode_steps):
        run.step()
    run.check_scores()
    run.cache.qe_synchronize()
    run.assert_all_live()
    assert run.codes_checked > 0
    for tr in run.tracked:
        if tr.live:
            run.check_bf16_windows(tr)
    print(f"{name}: out err {run.max_out_err:.2e}, score rel err {run.max_score_err:.2e}, "
          f"codes {run.codes_checked}, ambiguous {run.ambiguous}")


@pytest.mark.parametrize("host", ["pinned", "pageable"])
def test_host_buffers_trajectory(host):
    """The same path with every input and output in host memory: the kernels read pinned new
    tokens and write pinned outputs in place, pageable buffers go through copies, queries and the
    prefill are copied in; every unit still follows the oracle."""
    wl = dataclasses.replace(CASES["d128_w32_g4"], name="host_" + host, n_layers=2, decode_steps=24)
    track = [(b, l, h) for b in range(wl.batch) for l in range(wl.n_layers) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, wl.n_layers, track, host=host)
    run.prefill()
    for _ in range(wl.decode_steps):
        run.step()
    run.check_scores()
    run.cache.qe_synchronize()
    run.assert_all_live()
    assert run.codes_checked > 0 and run.route_events == wl.decode_steps // wl.route_period
    print(f"host {host}: out err {run.max_out_err:.2e}, score rel err {run.max_score_err:.2e}, "
          f"codes {run.codes_checked}")


ROPE_CASES = {
    "rope_d128_w32_g4": dataclasses.replace(CASES["d128_w32_g4"], name="rope_d128_w32_g4", rope_theta=10000.0,
                                            prefill=700, seed=41),
    "rope_d64_w16_g2": dataclasses.replace(CASES["d64_w64_g2"], name="rope_d64_w16_g2", window=16, route_period=8,
                                           n_sink=3, rope_theta=500.0, seed=42),
}


@pytest.mark.parametrize("name", sorted(ROPE_CASES))
def test_pre_rope_keys_trajectory(name):
    """Keys stored pre-RoPE (bf16 windows, 2-bit codes and the host store), rotated at their
    original positions inside the attention: every unit follows the oracle, which rotates the
    same stored keys in float64."""
    wl = ROPE_CASES[name]
    track = [(b, l, h) for b in range(wl.batch) for l in range(wl.n_layers) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, wl.n_layers, track)
    run.prefill()
    for _ in range(wl.decode_steps):
        run.step()
    run.check_scores()
    run.cache.qe_synchronize()
    run.assert_all_live()
    assert run.codes_checked > 0
    for tr in run.tracked:
        if tr.live:
            run.check_bf16_windows(tr)
    print(f"{name}: out err {run.max_out_err:.2e}, score rel err {run.max_score_err:.2e}, codes {run.codes_checked}")
