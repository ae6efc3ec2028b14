"""Full-size sampled parity on the 32-layer workloads (GPU).

Each test holds a whole workload in the cache and checks a few sampled units against the oracle.
The headline one is the 32K-context throughput workload: 32 layers, batch 16, GQA 32q/8kv, d 128,
32,768-token prefill, w 32, Omega 32, 8 % bf16 / 25 % 2-bit tokens. It is driven in the launch
configuration the benchmark times:

- direct calls up to the first routing event;
- then one decode step of the whole stack captured as a CUDA graph, plus a variant that ends
  with the routing event, replayed with fresh inputs in fixed buffers.

The oracle rebuilds only a few sampled units (batch element, layer, KV head) from the seeded
generator. For those units the test compares:

- attention outputs, every step;
- window scores and tiers, at each routing event (the first direct, the second inside a
  replayed graph);
- every 2-bit window's codes and parameters, bit for bit;
- every Full window's bf16 contents.

The Llama-shaped byte-budget stack (all 256 steps, 16 routing events) and the 131K-context
workload (one routing event over about 2,050 candidate windows per unit) run with direct calls.
"""
import numpy as np
import pytest

import qe_inputs as gen
from qe_testlib import OUT_TOL, ParityRun

pytestmark = pytest.mark.gpu

# first / last layer, first / last batch element and KV head, and one unit in between
SAMPLED = [(0, 0, 0), (5, 17, 3), (15, 31, 7)]


def test_throughput_32k_sampled_units_graph_replay():
    import torch
    wl = gen.WORKLOADS["throughput_32k"]
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(dev)          # capturable stream for the whole run
    torch.cuda.set_stream(stream)
    run = ParityRun(wl, wl.batch, wl.n_layers, SAMPLED, device_inputs=True)
    run.prefill()
    omega = wl.route_period
    for _ in range(omega):                   # direct calls through the first routing event
        run.step()
    assert run.route_events == 1

    Lyr, B, D = wl.n_layers, wl.batch, wl.head_dim
    kin = torch.empty(Lyr, B, wl.n_kv_heads, 1, D, device=dev, dtype=torch.int16)
    vin = torch.empty_like(kin)
    qin = torch.empty(Lyr, B, wl.n_q_heads, D, device=dev, dtype=torch.int16)
    out = torch.empty(Lyr, B, wl.n_q_heads, D, device=dev, dtype=torch.float32)
    cache = run.cache
    graphs = {}
    for routed in (False, True):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for layer in range(Lyr):
                cache.qe_append(layer, kin[layer], vin[layer], 1)
                cache.qe_decode_step(layer, qin[layer], out[layer])
            if routed:
                cache.qe_route(-1)
        graphs[routed] = g
    cache.qe_layer_info_sync()

    for _ in range(omega):                   # graph replays through the second routing event
        run.t += 1
        t = run.t
        pos = wl.prefill + t - 1
        for layer in range(Lyr):
            run.gdev.keys_values(layer, pos, 1, kin[layer], vin[layer], stream.cuda_stream)
            run.gdev.queries(layer, t, qin[layer], stream.cuda_stream)
        routed = t % omega == 0
        graphs[routed].replay()
        torch.cuda.synchronize(dev)
        got = out.cpu().numpy()
        for tr in run.tracked:
            if not tr.live:
                continue
            heads = range(tr.kvh * wl.group, (tr.kvh + 1) * wl.group)
            q = gen.bf16_bits_to_f32(gen.gen_queries(wl, tr.b, tr.layer, heads, t))
            kb, vb = gen.gen_keys_values(wl, tr.b, tr.layer, tr.kvh, pos, 1)
            o_ref, _, _ = tr.unit.decode_step(q, gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb))
            for i, h in enumerate(heads):
                err = np.linalg.norm(got[tr.layer, tr.b, h].astype(np.float64) - o_ref[i]) / np.linalg.norm(o_ref[i])
                run.max_out_err = max(run.max_out_err, err)
                assert err <= OUT_TOL, f"step {t} unit {(tr.b, tr.layer, tr.kvh)} head {h}: rel-L2 {err:.3e}"
        if routed:
            run.route_and_check(gpu_routed=True)
    assert run.route_events == 2

    full_checked = 0
    for tr in run.tracked:
        if tr.live:
            full_checked += run.check_bf16_windows(tr)
    info = cache.layer_info(0)
    assert (info.n_full, info.n_quant) == (info.kf, info.kq)
    print(f"full-size sampled parity: max out rel-L2 {run.max_out_err:.2e}, max score rel {run.max_score_err:.2e}, "
          f"2-bit windows compared {run.codes_checked}, Full windows compared {full_checked}, "
          f"tie-ambiguous units {run.ambiguous} {[tr.note for tr in run.tracked if tr.note]}")
    run.assert_all_live()
    assert run.codes_checked > 0 and full_checked > 0


def _direct_trajectory(wl, track, steps):
    """Drive the whole workload with direct calls for `steps` decode steps, comparing the
    sampled units every step and at every routing event; returns the run."""
    import torch
    dev = torch.device("cuda:0")
    torch.cuda.set_stream(torch.cuda.Stream(dev))
    run = ParityRun(wl, wl.batch, wl.n_layers, track, device_inputs=True)
    run.prefill()
    for _ in range(steps):
        run.step()
    return run


def test_llama8b_stack_byte_budget_sampled_units():
    """32 layers, GQA 32q/8kv, d 128, batch 1, 512-token prefill and all 256 decode steps, w 16,
    Omega 16 (16 routing events), 20 % KV byte budget with 10 % of tokens bf16."""
    wl = gen.WORKLOADS["llama8b_stack"]
    run = _direct_trajectory(wl, [(0, 0, 0), (0, 13, 5), (0, 31, 7)], wl.decode_steps)
    assert run.route_events == wl.decode_steps // wl.route_period
    full_checked = sum(run.check_bf16_windows(tr) for tr in run.tracked if tr.live)
    print(f"llama8b_stack: max out rel-L2 {run.max_out_err:.2e}, max score rel {run.max_score_err:.2e}, "
          f"2-bit windows compared {run.codes_checked}, Full windows {full_checked}, "
          f"tie-ambiguous {run.ambiguous} {[tr.note for tr in run.tracked if tr.note]}")
    run.assert_all_live()
    assert run.codes_checked > 0


def test_long_131k_sampled_units():
    """32 layers, GQA 32q/8kv, d 128, batch 1, 131,072-token prefill, w 64, Omega 64, 5 % bf16 /
    30 % 2-bit tokens: the routing event at step 64 ranks about 2,050 candidate windows per unit;
    eight more steps attend over the routed cache."""
    import dataclasses
    wl = dataclasses.replace(gen.WORKLOADS["long_131k"], decode_steps=72)
    run = _direct_trajectory(wl, [(0, 0, 0), (0, 31, 7)], 72)
    assert run.route_events == 1
    full_checked = sum(run.check_bf16_windows(tr) for tr in run.tracked if tr.live)
    info = run.cache.layer_info(31)
    assert (info.n_full, info.n_quant) == (info.kf, info.kq)
    print(f"long_131k: max out rel-L2 {run.max_out_err:.2e}, max score rel {run.max_score_err:.2e}, "
          f"2-bit windows compared {run.codes_checked}, Full windows {full_checked}, Kf {info.kf}, Kq {info.kq}, "
          f"tie-ambiguous {run.ambiguous}")
    run.assert_all_live()
    assert run.codes_checked > 0


def test_throughput_32k_pre_rope_sampled_units():
    """The 32K throughput workload with keys stored pre-RoPE (rotary base 10000): 40 steps of
    direct calls through the first routing event, three sampled units against the oracle."""
    import dataclasses
    wl = dataclasses.replace(gen.WORKLOADS["throughput_32k_rope"], decode_steps=40)
    run = _direct_trajectory(wl, SAMPLED, 40)
    assert run.route_events == 1
    full_checked = sum(run.check_bf16_windows(tr) for tr in run.tracked if tr.live)
    print(f"throughput_32k_rope: max out rel-L2 {run.max_out_err:.2e}, max score rel {run.max_score_err:.2e}, "
          f"2-bit windows compared {run.codes_checked}, Full windows {full_checked}")
    run.assert_all_live()
    assert run.codes_checked > 0
