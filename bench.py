"""Decode throughput of the tiered KV cache on the headline workload.

One step = one decode token for the whole stack: for every layer, append the new K/V,
run the attention with fused window scoring (qe_decode_attn + qe_attn_combine), and every
Omega steps route all layers (segmented top-K, packing, moves).  Inputs are seeded synthetic
tensors with the workload's shapes (qe_inputs), generated on the device before the timed
region; the cache per layer (~280 MB) and per step (~8.9 GB) is far larger than L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (the only other
implementation of this path) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and attn HBM GB/s vs peak; GQA 32q/8kv d128, 32K ctx"


def _peaks(key="hbm_gbs", fallback=6800.0):
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p[key]), "measured"
    except Exception:
        return fallback, "fallback"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, world


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the job ends when its slowest rank does)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: float, world: int, ms: float) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms / 1e3)


def workload_config(wl, world: int) -> dict:
    """The `config` object of the JSON line (shared by both arms)."""
    c = {
        "workload": wl.name, "batch": wl.batch, "context": wl.prefill, "layers": wl.n_layers,
        "q_heads": wl.n_q_heads, "kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim, "window": wl.window,
        "route_period": wl.route_period, "bf16_token_share": wl.frac_bf16, "int2_token_share": wl.frac_int2,
        "n_sink": wl.n_sink, "n_recent": wl.n_recent, "parallelism": f"replicas{world}",
    }
    if getattr(wl, "tiering", "windows") == "tokens":
        del c["window"]
        c.update({"tiering": "per-token five tiers", "int4_token_share": wl.frac_int4,
                  "nq1_token_share": wl.frac_nq1, "score_window": wl.score_window})
    return c


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples go to $QE_CLOCKS_DIR (default: the temp directory); the JSON line
        # carries their summary
        self.path = os.path.join(os.environ.get("QE_CLOCKS_DIR", tempfile.gettempdir()), f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------- ncu traffic record
# the sources each attention kernel is built from: its translation unit and the local headers it
# includes (the ncu record names the same list and their joint sha256)
KERNEL_SOURCES = {
    "qe_decode_attn": ["qe_attn.cu", "qe_kernels.cuh", "qe_partition.cuh", "qe_common.cuh"],
    "tk_attn": ["qe_tok.cu", "qe_exact_stats.cuh", "qe_tok.cuh", "qe_tok_kernels.h", "qe_common.cuh"],
}


def kernel_sources_sha256(kernel: str) -> str:
    """sha256 of the kernel's sources with comments removed and whitespace runs collapsed: an
    edit of a comment does not void the counters, an edit of the code does."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        src = open(os.path.join(ROOT, "tiered_quantize_evict_gb300", "csrc", name)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()


def _traffic(workload: str, kernel: str = "qe_decode_attn"):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, if the
    kernel's sources are unchanged since it was captured (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_files") != KERNEL_SOURCES[kernel]:
            return None
        if rec.get("source_sha256") != kernel_sources_sha256(kernel):
            return None
        return rec.get("dram_bytes_per_launch_full")
    except Exception:
        return None


def _route_counts(cache):
    """Cumulative routing counters of all layers (window tiering), or None."""
    try:
        st = cache.route_stats(-1)
    except Exception:
        return None
    return {f: int(getattr(st, f)) for f in ("first_packs", "ledger_reuses", "promotions", "evictions",
                                            "bf16_reclaims", "int2_reclaims", "ledger_writes")}


# ---------------------------------------------------------------------------- our implementation
def run_ours(args):
    import torch
    import torch.distributed as dist

    import qe_inputs as gen
    import qe_inputs.cuda as gcuda
    import tiered_quantize_evict_gb300 as qe

    rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = gen.WORKLOADS[args.workload]
    if args.layers or args.batch:          # profiling cases only: smaller stack, same per-layer shapes
        import dataclasses
        wl = dataclasses.replace(wl, n_layers=args.layers or wl.n_layers, batch=args.batch or wl.batch)
    B, Lyr, Hq, Hkv, D = wl.batch, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    omega = wl.route_period
    K, W = args.steps, args.warmup
    NQ = max(1, args.verify)          # tokens per step: a speculative verify of NQ drafts, all kept
    verify = args.verify > 0

    def routes_at(t):
        return (t * NQ) // omega > ((t - 1) * NQ) // omega

    def next_route_step(t):           # first step >= t that ends with a routing event
        while not routes_at(t):
            t += 1
        return t

    pre = next_route_step(1)          # steps through the first routing event
    # The warm-up ends with a routing event, so the timed region starts right after one and each
    # whole Omega-token period inside it holds exactly one event.
    W_eff = next_route_step(pre + W) - pre
    P = next_route_step(pre + 1) - pre          # steps between routing events
    KR = max(K, P)                              # per-launch timing leg: sees at least one event
    # steps: pre-roll, warm-up, K timed, KR per-launch timing, up to P aligning, K end to end
    total_steps = pre + W_eff + K + KR + P + K
    max_ctx = wl.prefill + max(wl.decode_steps, (total_steps + pre + 1) * NQ)
    stream = torch.cuda.Stream(dev)     # capturable: all work of this run is ordered on it
    torch.cuda.set_stream(stream)
    cache = qe.QECache(qe.config_from_workload(wl, max_context=max_ctx), stream.cuda_stream)
    if verify:
        vpath = {"auto": 0, "fused": 1, "per_draft": 2}[args.verify_path]
        assert qe.debug_inject(qe.QE_DEBUG_VERIFY_PATH, vpath, cache) == qe.QE_OK
    g = gcuda.DeviceGenerator(wl, device=dev)

    # prefill, one layer at a time (2 x B x Hkv x L0 x d bf16 = 2 GB per layer)
    kbuf = torch.empty(B, Hkv, wl.prefill, D, device=dev, dtype=torch.int16)
    vbuf = torch.empty_like(kbuf)
    for layer in range(Lyr):
        g.keys_values(layer, 0, wl.prefill, kbuf, vbuf, stream.cuda_stream)
        cache.qe_append(layer, kbuf, vbuf, wl.prefill)
    cache.qe_synchronize()
    del kbuf, vbuf
    torch.cuda.empty_cache()

    # per-step inputs, device resident
    def make_inputs(t):
        """Inputs of step t (1-based): tokens (t-1) NQ + j and their queries, j < NQ."""
        if not verify:
            k = torch.empty(Lyr, B, Hkv, 1, D, device=dev, dtype=torch.int16)
            v = torch.empty_like(k)
            q = torch.empty(Lyr, B, Hq, D, device=dev, dtype=torch.int16)
            for layer in range(Lyr):
                g.keys_values(layer, wl.prefill + t - 1, 1, k[layer], v[layer], stream.cuda_stream)
                g.queries(layer, t, q[layer], stream.cuda_stream)
            return k, v, q
        k = torch.empty(Lyr, NQ, B, Hkv, D, device=dev, dtype=torch.int16)   # draft-major
        v = torch.empty_like(k)
        q = torch.empty(Lyr, NQ, B, Hq, D, device=dev, dtype=torch.int16)
        for layer in range(Lyr):
            for j in range(NQ):
                i = (t - 1) * NQ + j
                g.keys_values(layer, wl.prefill + i, 1, k[layer, j].view(B, Hkv, 1, D),
                              v[layer, j].view(B, Hkv, 1, D), stream.cuda_stream)
                g.queries(layer, i + 1, q[layer, j], stream.cuda_stream)
        return k, v, q

    out = torch.empty(NQ, B, Hq, D, device=dev, dtype=torch.float32) if verify else \
        torch.empty(B, Hq, D, device=dev, dtype=torch.float32)

    def step(t, k, v, q, o=out, route_events=None):
        for layer in range(Lyr):
            if verify:
                cache.qe_verify(layer, q[layer], k[layer], v[layer], o, NQ)
                cache.qe_verify_commit(layer, NQ)
            else:
                cache.qe_append(layer, k[layer], v[layer], 1)
                cache.qe_decode_step(layer, q[layer], o)
        if routes_at(t):
            if route_events is not None:      # CUDA events around the routing call of all layers
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record(stream)
                cache.qe_route(-1)
                ev[1].record(stream)
                route_events.append((t, ev))
            else:
                cache.qe_route(-1)

    t = 0
    for _ in range(pre + W_eff):        # pre-roll through the first routing event, then warm-up
        t += 1
        k, v, q = make_inputs(t)
        step(t, k, v, q)
    cache.qe_synchronize()
    t_timed0 = t + 1

    # The K timed decode steps of the whole stack captured as one CUDA graph and launched once:
    # every step's inputs sit in their own device buffers, as a model's projections would leave
    # them, and all launch arguments are step-invariant apart from those buffers (the kernels
    # read the layer state from device memory), so the timed region has no host involvement.
    timed = [make_inputs(t + 1 + i) for i in range(K)]
    torch.cuda.synchronize(dev)
    n_routes = 0
    launches_before = cache.kernel_launches()
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream, capture_error_mode="thread_local"):
        for i in range(K):
            tt = t + 1 + i
            step(tt, *timed[i])
            n_routes += routes_at(tt)
    graph_launches = cache.kernel_launches() - launches_before   # kernels the graph holds
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g_all.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t += K
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_total = e0.elapsed_time(e1)
    launches = graph_launches
    cache.qe_synchronize()
    cache.qe_layer_info_sync()
    del timed

    # per-launch attention times: the same step, launched directly with CUDA events around
    # every qe_decode_attn launch on the handle's stream, and around every routing call
    rl = [make_inputs(t + 1 + i) for i in range(KR)]
    torch.cuda.synchronize(dev)
    route_events = []
    rs0 = _route_counts(cache)
    cache.set_timing(True)
    for i in range(KR):
        t += 1
        step(t, *rl[i], route_events=route_events)
    torch.cuda.synchronize(dev)
    cache.set_timing(False)
    attn_ms, attn_launches, attn_bytes = cache.timing()
    # the launch and event overhead inside each of those event times: an empty launch of the
    # same shape between the same events (window path; the five-tier launch has its own shape)
    overhead_us = None
    if getattr(wl, "tiering", "windows") != "tokens" and not verify:
        overhead_us = cache.launch_overhead(200)
    rs1 = _route_counts(cache)
    route_ms = [a.elapsed_time(b) for _, (a, b) in route_events]
    route_steps = [ts * NQ for ts, _ in route_events]
    cache.qe_synchronize()
    del rl

    # align: the end-to-end leg, like the timed one, starts right after a routing event
    if not routes_at(t):
        for _ in range(next_route_step(t) - t):
            t += 1
            step(t, *make_inputs(t))
    cache.qe_synchronize()
    step_e2e0 = t + 1
    e2e_routes = sum(routes_at(t + 1 + i) for i in range(K))

    # end to end through the C ABI with host buffers: pinned inputs copied in and the
    # outputs read back every step, inside the timed region
    host_in = []
    for i in range(K):
        k, v, q = make_inputs(t + 1 + i)
        host_in.append((k.cpu().pin_memory(), v.cpu().pin_memory(), q.cpu().pin_memory()))
    host_out = torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in[0])
    d2h = host_out.numel() * host_out.element_size() * Lyr
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    t_e2e0 = time.perf_counter()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for i in range(K):
        t += 1
        step(t, *host_in[i], o=host_out)
    e3.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max(e2.elapsed_time(e3), (time.perf_counter() - t_e2e0) * 1e3)
    cache.qe_synchronize()

    # Routing belongs to every step (one event per Omega tokens).  A timed region of K steps that
    # starts right after an event holds floor(K NQ / Omega) of them; when K is not a whole
    # number of periods, the missing fraction of an event is added at the measured mean cost
    # of the events of the per-launch leg.
    per_k = K * NQ / omega
    route_mean = sum(route_ms) / len(route_ms) if route_ms else 0.0
    graph_ms = ms_total
    add_ms = max(0.0, per_k - n_routes) * route_mean
    add_e2e_ms = max(0.0, per_k - e2e_routes) * route_mean
    ms_total = graph_ms + add_ms
    e2e_ms = e2e_ms + add_e2e_ms
    ms_total = max_over_ranks(ms_total, world, dev)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    value = whole_job_rate(B * NQ * K, world, ms_total)
    e2e_val = whole_job_rate(B * NQ * K, world, e2e_ms)
    peak, peak_kind = _peaks()
    achieved = attn_bytes / (attn_ms / 1e3) / 1e9 if attn_ms > 0 else None
    info = cache.layer_info(0)
    tok = getattr(wl, "tiering", "windows") == "tokens"
    if tok:
        cnt = cache.token_counts(0).mean(axis=0)
        kv_unit = {"bf16_ranked": round(float(cnt[0]), 1), "int4": round(float(cnt[1]), 1),
                   "int2": round(float(cnt[2]), 1), "nq1": round(float(cnt[3]), 1), "bf16_tail": round(float(cnt[4]), 1)}
    else:
        kv_unit = {"full": info.n_full, "quant": info.n_quant, "pinned": info.n_pinned}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_total / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded qe_inputs generator, device-side)",
        "config": {
            **workload_config(wl, world),
            "timed_decode_steps": [t_timed0, t_timed0 + K - 1],
            "launch": ("the K timed steps as one CUDA graph (per step %d layers x token append, attention, merge; "
                       "re-rank every Omega), started right after a re-rank" % Lyr) if tok else
                      ("the K timed steps as one CUDA graph (per step %d layers x attention with the token "
                       "append, combine; routing every Omega), started right after a routing event" % Lyr),
            "routing_in_value": {
                "events_per_K_steps_at_one_per_Omega": round(per_k, 4),
                "events_in_timed_graph": n_routes,
                "added_ms_for_missing_fraction": round(add_ms, 4),
                "graph_ms": round(graph_ms, 4),
                "rule": "value = tokens / (graph time + (K NQ / Omega - events in the graph) x mean measured "
                        "event time); the timed graph starts right after an event, so it holds the whole "
                        "periods' events itself and only a partial period is added"},
            ("kv_tokens_per_layer_unit" if tok else "kv_per_layer_unit"): kv_unit,
            "l2": "inputs larger than L2: %.0f MB read per layer launch, %.1f GB per step (a layer's data is "
                  "read again only after the other layers' data)" % (info.attn_bytes / 1e6, info.attn_bytes * Lyr / 1e9),
            "kv_dtypes": ("bf16 + per-token 4/2-bit uniform and 1-bit normal codes (fp32 params); fp32 accumulate"
                          if tok else "bf16 tiles + 2-bit codes (fp32 min/scale); fp32 accumulate"),
        },
        "roofline": {
            "bound": "hbm", "kernel": "tk_attn" if tok else "qe_decode_attn", "achieved": round(achieved, 1) if achieved else None,
            "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4) if achieved else None,
            "traffic": _traffic(wl.name, "tk_attn" if tok else "qe_decode_attn"),
            "algorithmic_bytes_per_launch": round(attn_bytes / max(attn_launches, 1)),
            "avg_launch_us": round(attn_ms * 1e3 / max(attn_launches, 1), 2),
            "attn_share_of_step": round((attn_ms / KR) / (ms_total / K), 4) if ms_total > 0 else None,
            "measured_on": "the next %d decode steps launched directly, CUDA events around each launch" % KR,
            # the event times hold launch and event overhead; measured, not subtracted above
            "event_overhead_us": round(overhead_us, 2) if overhead_us is not None else None,
            "frac_without_event_overhead": (
                round(attn_bytes / max(attn_launches, 1) / ((attn_ms * 1e3 / max(attn_launches, 1) - overhead_us) * 1e-6)
                      / 1e9 / peak, 4)
                if overhead_us is not None and attn_ms > 0 and attn_ms * 1e3 / max(attn_launches, 1) > overhead_us
                else None),
            "event_overhead_measured_on": "200 empty launches of the attention launch's shape (grid, block, dynamic "
                                          "shared memory, programmatic serialization) between two events each, "
                                          "same stream, same run (qe_launch_overhead)",
        },
        "routing": {
            "events": len(route_ms),
            "at_decode_steps": route_steps,
            "ms_per_event": [round(x, 3) for x in route_ms],
            "ms_per_step_amortized": round(sum(route_ms) / K, 4),
            "counts": {kk: rs1[kk] - rs0[kk] for kk in rs1} if rs0 and rs1 else None,
            "measured_on": ("%d direct-launch steps after the timed ones, CUDA events around each qe_route(-1) "
                            "call (every layer's %s and moves)" % (KR, "re-rank" if tok else "routing")),
        },
        "e2e": {"value": round(e2e_val, 2), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "decode_steps": [step_e2e0, step_e2e0 + K - 1],
                "routing_events_timed": e2e_routes, "added_ms_for_missing_fraction": round(add_e2e_ms, 4),
                "path": "direct C-ABI calls on pinned host buffers: queries copied in, new K/V read "
                        "and outputs written in place by the kernels over the host link"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    # a verify on the fused path: its attention launch is the tensor-core contraction
    G = Hq // Hkv
    fused = verify and (args.verify_path == "fused" or (args.verify_path == "auto" and NQ >= 5)) \
        and not wl.rope_theta and NQ * G <= 64
    if fused:
        tokens = B * Hkv * ((info.n_full + info.n_quant + info.n_pinned) * wl.window + wl.n_sink)
        flops = 4.0 * NQ * G * D * tokens   # Q K^T and P V per attended token and query row
        avg_s = attn_ms / 1e3 / max(attn_launches, 1)
        tpeak, tpeak_kind = _peaks("bf16_tflops", 1900.0)
        t_ach = flops / avg_s / 1e12 if attn_ms > 0 else None
        line["roofline"] = {
            "bound": "tensor", "kernel": "qe_verify_attn", "achieved": round(t_ach, 2) if t_ach else None,
            "peak": tpeak, "peak_kind": tpeak_kind + " (dense bf16, burst)", "unit": "TFLOP/s",
            "frac": round(t_ach / tpeak, 4) if t_ach else None, "traffic": None,
            "algorithmic_flops_per_launch": flops,
            "flops_rule": "4 R d per attended token (Q K^T and P V), R = drafts x G rows; tokens = the kept "
                          "windows of every unit (the 2-bit keys' three exact bf16 parts and P's two are not "
                          "counted)",
            "avg_launch_us": round(avg_s * 1e6, 2),
            "attn_gbs": round(achieved, 1) if achieved else None,
            "measured_on": "the next %d verify steps launched directly, CUDA events around each fused attention "
                           "launch" % KR,
        }
    if verify:
        line["config"]["verify"] = {
            "drafts_per_step": NQ, "accepted": "all", "path": args.verify_path,
            "step": "per layer qe_verify of the drafts (each draft query attends over the cache and the "
                    "drafts before it; masses held per query) then qe_verify_commit; value counts every draft"}
    cache.close()
    if world > 1:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------------------- the oracle on host cores
def _oracle_worker(a):
    """Set one unit up to its steady state (untimed), then time `steps` decode steps."""
    name, b, layer, kvh, n_steps, first_step = a
    import numpy as np
    import qe_inputs as gen
    from oracle.run import make_unit, prefill, step_inputs
    wl = gen.WORKLOADS[name]
    unit = make_unit(wl, max_context=wl.prefill + first_step + n_steps + 1)
    prefill(wl, unit, b, layer, kvh)
    routes = hasattr(unit, "route")          # window tiers route explicitly; token tiers re-rank in the step
    for t in range(1, first_step):
        q, k, v = step_inputs(wl, b, layer, kvh, t)
        unit.decode_step(q, k, v)
        if routes and t % wl.route_period == 0:
            unit.route()
    times = []
    for t in range(first_step, first_step + n_steps):
        q, k, v = step_inputs(wl, b, layer, kvh, t)
        t0 = time.perf_counter()
        unit.decode_step(q, k, v)
        if routes and t % wl.route_period == 0:
            unit.route()
        times.append(time.perf_counter() - t0)
    return times


def oracle_baseline(workload: str, n_units: int, n_steps: int, n_warm: int = 0):
    """Tokens/s of the CPU oracle extrapolated from a bounded sample of units.

    Each sampled unit runs `n_warm` untimed and then `n_steps` timed decode steps.
    """
    import multiprocessing as mp

    import qe_inputs as gen
    wl = gen.WORKLOADS[workload]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    units_total = wl.batch * wl.n_layers * wl.n_kv_heads
    n_units = max(1, min(n_units, units_total))      # distinct units (the stride is prime)
    first = wl.route_period + 1
    jobs = []
    for i in range(n_units):
        u = (i * 2654435761) % units_total
        b, rest = divmod(u, wl.n_layers * wl.n_kv_heads)
        layer, kvh = divmod(rest, wl.n_kv_heads)
        jobs.append((workload, b, layer, kvh, n_warm + n_steps, first))
    workers = min(cores, n_units)
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        res = pool.map(_oracle_worker, jobs)
    per_unit_step = sum(sum(r[n_warm:]) for r in res) / (n_units * n_steps)   # seconds, one core
    step_s = per_unit_step * units_total / workers                       # all units, `workers` cores
    # what one step of the sample itself took: the units run side by side, one per core
    sample_step_s = max(sum(r[n_warm:]) for r in res) / n_steps * math.ceil(n_units / workers)
    return {"value": round(wl.batch / step_s, 4), "unit": "tokens/s", "cores": workers, "kind": "oracle",
            "extrapolated": True, "sample_ms_per_step": round(sample_step_s * 1e3, 3),
            "extrapolated_ms_per_step": round(step_s * 1e3, 3),
            "sample": f"{n_units} units x {n_steps} timed steady-state decode steps (after the first routing "
                      f"event and {n_warm} untimed warm-up steps) of {workload}, extrapolated to all "
                      f"{units_total} units on {workers} cores; setup (prefill, pre-roll, first route) untimed"}, \
        step_s, sample_step_s


def run_reference(args):
    rank, world = _dist()
    if rank != 0:
        return None
    import qe_inputs as gen
    wl = gen.WORKLOADS[args.workload]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    # each step: one decode step of `cores` sampled units (bounded sample of the workload)
    n_units = max(1, min(cores, 16))
    t0 = time.perf_counter()
    base, step_s, sample_step_s = oracle_baseline(args.workload, n_units, args.steps, n_warm=args.warmup)
    wall = time.perf_counter() - t0
    v = base["value"]
    # ms_per_step is what one step of the bounded sample took here (the run's own clock);
    # value is the whole workload's rate extrapolated from it (cpu_baseline.extrapolated_ms_per_step)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sample_step_s * 1e3, 3),
            "extrapolated": True, "extrapolated_ms_per_step": round(step_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded qe_inputs generator)",
            "config": workload_config(wl, world),
            "cpu_baseline": base,
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="throughput_32k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="profiling only: fewer layers than the workload")
    ap.add_argument("--batch", type=int, default=0, help="profiling only: other batch than the workload")
    ap.add_argument("--verify", type=int, default=0,
                    help="steps are speculative verifies of this many drafts per layer, all accepted")
    ap.add_argument("--verify-path", choices=["auto", "fused", "per_draft"], default="auto",
                    help="qe_verify's path (QE_DEBUG_VERIFY_PATH): automatic, the fused tensor-core "
                         "launch, or one decode step per draft")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world = _dist()
    if args.impl == "reference":
        line = run_reference(args)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line = run_ours(args)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            base, _, _ = oracle_baseline(args.workload, n_units=min(16, len(os.sched_getaffinity(0))), n_steps=2)
            line["cpu_baseline"] = base
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
