"""Five-tier per-token cache (HqeKV reading notes) on the GPU against the oracle, every unit of
small workloads through whole trajectories.

Each decode step compares every unit's attention outputs.  At each re-rank the test compares:
- every position's score;
- the tiers after both sides re-rank on the GPU's scores;
- every quantized token's codes and float32 parameters, bit for bit;
- every BF16 token's values.

Ranking parity is asserted on identical scores: the GPU's float32 scores are handed to the oracle
before it re-ranks, because near-ties make both rankings correct when the scores differ in the
last bits.
"""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from oracle import hqekv as H
from oracle.run import make_unit
from qe_testlib import OUT_TOL, SCORE_ATOL, SCORE_RTOL, host_kv, host_q, to_dev, torch_dev

pytestmark = pytest.mark.gpu

BASE = gen.WORKLOADS["tiny_hqe"]
CASES = {
    "d128_g4": BASE,
    "d64_g2_m0": dataclasses.replace(BASE, name="d64_g2_m0", head_dim=64, n_q_heads=6, n_kv_heads=3, batch=1,
                                     prefill=203, decode_steps=40, route_period=10, score_window=0, n_sink=3,
                                     n_recent=9, seed=31),
    "d128_g1_long_window": dataclasses.replace(BASE, name="d128_g1", n_q_heads=2, n_kv_heads=2, batch=2, n_layers=1,
                                               prefill=520, decode_steps=36, route_period=12, score_window=12,
                                               frac_bf16=0.05, frac_int4=0.15, frac_int2=0.25, frac_nq1=0.45,
                                               seed=32),
}


class TokRun:
    def __init__(self, wl, host=None):
        """host: None (device buffers), "pinned" or "pageable": where every call's inputs and
        outputs live."""
        import tiered_quantize_evict_gb300 as qe
        torch, dev = torch_dev()
        self.host = host
        self.torch, self.dev, self.wl = torch, dev, wl
        self.cache = qe.QECache(qe.config_from_workload(wl), torch.cuda.current_stream().cuda_stream)
        self.units = {(b, l, h): make_unit(wl) for b in range(wl.batch) for l in range(wl.n_layers)
                      for h in range(wl.n_kv_heads)}
        self.t = 0
        self.max_out = 0.0
        self.max_score = 0.0
        self.codes_checked = 0
        self.bf16_checked = 0
        if host == "pinned":
            self.out = torch.empty(wl.batch, wl.n_q_heads, wl.head_dim, dtype=torch.float32).pin_memory()
        elif host == "pageable":
            self.out = np.zeros((wl.batch, wl.n_q_heads, wl.head_dim), np.float32)
        else:
            self.out = torch.empty(wl.batch, wl.n_q_heads, wl.head_dim, device=dev, dtype=torch.float32)

    def place(self, a):
        a = np.ascontiguousarray(a).view(np.int16)
        if self.host == "pinned":
            return self.torch.from_numpy(a).pin_memory()
        if self.host == "pageable":
            return a.copy()
        return to_dev(a)

    def read_out(self):
        if self.host:
            self.cache.qe_synchronize()
            return np.array(self.out, dtype=np.float64) if self.host == "pageable" else self.out.numpy().astype(np.float64)
        return self.out.cpu().numpy().astype(np.float64)

    def u_index(self, b, h):
        return b * self.wl.n_kv_heads + h

    def prefill(self):
        wl = self.wl
        for layer in range(wl.n_layers):
            K, V = host_kv(wl, layer, 0, wl.prefill, wl.batch)
            kt, vt = self.place(K), self.place(V)
            self.cache.qe_append(layer, kt, vt, wl.prefill)
            self.cache.qe_synchronize()
            for b in range(wl.batch):
                for h in range(wl.n_kv_heads):
                    self.units[(b, layer, h)].append(gen.bf16_bits_to_f32(K[b, h]), gen.bf16_bits_to_f32(V[b, h]))

    def step(self):
        wl = self.wl
        self.t += 1
        t = self.t
        pos = wl.prefill + t - 1
        for layer in range(wl.n_layers):
            K, V = host_kv(wl, layer, pos, 1, wl.batch)
            Q = host_q(wl, layer, t, wl.batch)
            kt, vt, qt = self.place(K), self.place(V), self.place(Q)   # alive until read_out syncs
            self.cache.qe_append(layer, kt, vt, 1)
            self.cache.qe_decode_step(layer, qt, self.out)
            got = self.read_out()
            for b in range(wl.batch):
                for h in range(wl.n_kv_heads):
                    heads = slice(h * wl.group, (h + 1) * wl.group)
                    q = gen.bf16_bits_to_f32(Q[b, heads])
                    o, _ = self.units[(b, layer, h)].decode_step(q, gen.bf16_bits_to_f32(K[b, h]),
                                                                 gen.bf16_bits_to_f32(V[b, h]), auto_rerank=False)
                    for i in range(wl.group):
                        err = np.linalg.norm(got[b, h * wl.group + i] - o[i]) / np.linalg.norm(o[i])
                        self.max_out = max(self.max_out, err)
                        assert err <= OUT_TOL, f"step {t} layer {layer} unit {(b, h)} head {i}: rel-L2 {err:.2e}"
        if t % wl.route_period == 0:
            self.rerank_and_check()

    def rerank_and_check(self):
        wl = self.wl
        for layer in range(wl.n_layers):
            S = self.cache.token_scores(layer)
            for b in range(wl.batch):
                for h in range(wl.n_kv_heads):
                    un = self.units[(b, layer, h)]
                    u = self.u_index(b, h)
                    live = (un.tier[:un.L] != H.EVICT) & (np.arange(un.L) >= wl.n_sink)
                    ref = un.S[:un.L][live].astype(np.float64)
                    got = S[u, :un.L][live].astype(np.float64)
                    err = np.abs(got - ref)
                    assert np.all(err <= SCORE_RTOL * ref + SCORE_ATOL), \
                        f"t {self.t} layer {layer} unit {u}: score error {err.max():.2e}"
                    self.max_score = max(self.max_score, float(np.max(err / np.maximum(ref, 1e-30))) if ref.size else 0)
                    un.S[:un.L] = np.where(np.arange(un.L) < wl.n_sink, 0, S[u, :un.L])   # route on the GPU's scores
        self.cache.qe_route(-1)
        for un in self.units.values():
            un.rerank()
        self.check_state()

    def check_state(self):
        wl = self.wl
        for layer in range(wl.n_layers):
            tiers = self.cache.token_tiers(layer)
            for b in range(wl.batch):
                for h in range(wl.n_kv_heads):
                    un = self.units[(b, layer, h)]
                    u = self.u_index(b, h)
                    ref = un.tier[:un.L]
                    bad = np.flatnonzero(tiers[u, :un.L] != ref)
                    assert bad.size == 0, f"t {self.t} layer {layer} unit {u}: tiers differ at {bad[:8].tolist()} " \
                                          f"(gpu {tiers[u, bad[:8]].tolist()}, oracle {ref[bad[:8]].tolist()})"
                    assert np.all(tiers[u, un.L:] == 255)
                    for p in range(un.L):
                        z = int(ref[p])
                        if z == H.EVICT:
                            continue
                        tier, kb, vb, kc, vc, par = self.cache.token(layer, u, p)
                        assert tier == z
                        if z == H.BF16:
                            if p % 7 == 0:   # a sample of the BF16 tokens
                                assert np.array_equal(gen.bf16_bits_to_f32(kb), un.K[p])
                                assert np.array_equal(gen.bf16_bits_to_f32(vb), un.V[p])
                                self.bf16_checked += 1
                            continue
                        tc = un.codes[p]
                        assert np.array_equal(kc, tc.k_codes), f"layer {layer} unit {u} pos {p} tier {z}: key codes"
                        assert np.array_equal(vc, tc.v_codes), f"layer {layer} unit {u} pos {p} tier {z}: value codes"
                        ref_par = np.array([tc.k_p0, tc.k_p1, tc.v_p0, tc.v_p1], np.float32)
                        assert np.array_equal(par.view(np.uint32), ref_par.view(np.uint32)), \
                            f"layer {layer} unit {u} pos {p} tier {z}: params {par} vs {ref_par}"
                        self.codes_checked += 1


@pytest.mark.parametrize("name", sorted(CASES))
def test_five_tier_trajectory(name):
    wl = CASES[name]
    run = TokRun(wl)
    run.prefill()
    run.check_state()
    for _ in range(wl.decode_steps):
        run.step()
    run.cache.qe_synchronize()
    counts = run.cache.token_counts(0)
    print(f"{name}: max out rel-L2 {run.max_out:.2e}, max score rel {run.max_score:.2e}, codes {run.codes_checked}, "
          f"bf16 {run.bf16_checked}, counts unit 0 {counts[0].tolist()}")
    assert run.codes_checked > 0
    assert (counts[:, 1:4] > 0).all()


@pytest.mark.parametrize("host", ["pinned", "pageable"])
def test_five_tier_host_buffers(host):
    """Host inputs and outputs: pinned tokens and queries are read, outputs written, in place by
    the kernels; pageable ones go through copies; the trajectory still follows the oracle."""
    wl = dataclasses.replace(CASES["d128_g4"], decode_steps=32)
    run = TokRun(wl, host=host)
    run.prefill()
    for _ in range(wl.decode_steps):
        run.step()
    run.cache.qe_synchronize()
    print(f"five-tier host {host}: max out rel-L2 {run.max_out:.2e}, codes {run.codes_checked}")
    assert run.codes_checked > 0


def test_hqe_16k_sampled_units_graph_replay():
    """The 16K five-tier workload at full size (32 layers, batch 8, GQA 32q/8kv, d 128, 16,384-token
    prefill, re-rank every 64 steps over the last 20 steps' attention), in the benchmark's launch
    configuration: direct calls through the first re-rank, then one decode step of the whole stack
    captured as a CUDA graph (plus the variant that ends with the re-rank) and replayed with fresh
    inputs.  Three sampled units follow the oracle: outputs every step, scores, tiers, codes and
    parameters at both re-ranks."""
    import torch
    import qe_inputs.cuda as gc
    import tiered_quantize_evict_gb300 as qe
    wl = gen.WORKLOADS["hqe_16k"]
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    cache = qe.QECache(qe.config_from_workload(wl), stream.cuda_stream)
    g = gc.DeviceGenerator(wl, device=dev)
    Lyr, B, D, Hq, Hkv = wl.n_layers, wl.batch, wl.head_dim, wl.n_q_heads, wl.n_kv_heads
    sampled = [(0, 0, 0), (3, 17, 5), (7, 31, 7)]
    units = {s: make_unit(wl) for s in sampled}
    kbuf = torch.empty(B, Hkv, wl.prefill, D, device=dev, dtype=torch.int16)
    vbuf = torch.empty_like(kbuf)
    for layer in range(Lyr):
        g.keys_values(layer, 0, wl.prefill, kbuf, vbuf, stream.cuda_stream)
        cache.qe_append(layer, kbuf, vbuf, wl.prefill)
    del kbuf, vbuf
    for (b, layer, h), un in units.items():
        kb, vb = gen.gen_keys_values(wl, b, layer, h, 0, wl.prefill)
        un.append(gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb))
    kin = torch.empty(Lyr, B, Hkv, 1, D, device=dev, dtype=torch.int16)
    vin = torch.empty_like(kin)
    qin = torch.empty(Lyr, B, Hq, D, device=dev, dtype=torch.int16)
    out = torch.empty(Lyr, B, Hq, D, device=dev, dtype=torch.float32)
    stats = {"out": 0.0, "score": 0.0, "codes": 0}

    def inputs(t):
        for layer in range(Lyr):
            g.keys_values(layer, wl.prefill + t - 1, 1, kin[layer], vin[layer], stream.cuda_stream)
            g.queries(layer, t, qin[layer], stream.cuda_stream)

    def compare(t):
        got = out.cpu().numpy().astype(np.float64)
        for (b, layer, h), un in units.items():
            heads = range(h * wl.group, (h + 1) * wl.group)
            q = gen.bf16_bits_to_f32(gen.gen_queries(wl, b, layer, heads, t))
            kb, vb = gen.gen_keys_values(wl, b, layer, h, wl.prefill + t - 1, 1)
            o, _ = un.decode_step(q, gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb), auto_rerank=False)
            for i, hq in enumerate(heads):
                err = np.linalg.norm(got[layer, b, hq] - o[i]) / np.linalg.norm(o[i])
                stats["out"] = max(stats["out"], err)
                assert err <= OUT_TOL, f"step {t} unit {(b, layer, h)} head {hq}: rel-L2 {err:.2e}"

    def scores_then_rerank(t, gpu_routed):
        for (b, layer, h), un in units.items():
            u = b * Hkv + h
            S = cache.token_scores(layer)[u]
            live = (un.tier[:un.L] != H.EVICT) & (np.arange(un.L) >= wl.n_sink)
            ref = un.S[:un.L][live].astype(np.float64)
            err = np.abs(S[:un.L][live] - ref)
            assert np.all(err <= SCORE_RTOL * ref + SCORE_ATOL), f"t {t} unit {(b, layer, h)}: score {err.max():.2e}"
            stats["score"] = max(stats["score"], float(np.max(err / np.maximum(ref, 1e-30))))
            un.S[:un.L] = np.where(np.arange(un.L) < wl.n_sink, 0, S[:un.L])
        if not gpu_routed:
            cache.qe_route(-1)
        for un in units.values():
            un.rerank()
        for (b, layer, h), un in units.items():
            u = b * Hkv + h
            tiers = cache.token_tiers(layer)[u]
            assert np.array_equal(tiers[:un.L], un.tier[:un.L]), f"t {t} unit {(b, layer, h)}: tiers"
            quant = [p for p in range(un.L) if un.tier[p] in (H.INT4, H.INT2, H.NQ1)]
            for p in quant[::37]:   # every 37th quantized token
                tier, _, _, kc, vc, par = cache.token(layer, u, p)
                tc = un.codes[p]
                assert tier == tc.tier and np.array_equal(kc, tc.k_codes) and np.array_equal(vc, tc.v_codes), \
                    f"t {t} unit {(b, layer, h)} pos {p}: codes"
                ref_par = np.array([tc.k_p0, tc.k_p1, tc.v_p0, tc.v_p1], np.float32)
                assert np.array_equal(par.view(np.uint32), ref_par.view(np.uint32)), f"pos {p}: params"
                stats["codes"] += 1

    omega = wl.route_period
    for t in range(1, omega + 1):            # direct calls through the first re-rank
        inputs(t)
        for layer in range(Lyr):
            cache.qe_append(layer, kin[layer], vin[layer], 1)
            cache.qe_decode_step(layer, qin[layer], out[layer])
        torch.cuda.synchronize(dev)
        compare(t)
        if t == omega:
            scores_then_rerank(t, gpu_routed=False)
    # one decode step of the stack and one re-rank of every layer, each captured once
    g_step, g_route = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream, capture_error_mode="thread_local"):
        for layer in range(Lyr):
            cache.qe_append(layer, kin[layer], vin[layer], 1)
            cache.qe_decode_step(layer, qin[layer], out[layer])
    with torch.cuda.graph(g_route, stream=stream, capture_error_mode="thread_local"):
        cache.qe_route(-1)
    for t in range(omega + 1, 2 * omega + 1):   # graph replays through the second re-rank
        inputs(t)
        g_step.replay()
        torch.cuda.synchronize(dev)
        compare(t)
        if t % omega == 0:
            cache.qe_layer_info_sync()
            g_route_run = lambda: g_route.replay()
            # scores before the re-rank go to the oracle, then the captured re-rank runs
            for (b, layer, h), un in units.items():
                u = b * Hkv + h
                S = cache.token_scores(layer)[u]
                live = (un.tier[:un.L] != H.EVICT) & (np.arange(un.L) >= wl.n_sink)
                ref = un.S[:un.L][live].astype(np.float64)
                err = np.abs(S[:un.L][live] - ref)
                assert np.all(err <= SCORE_RTOL * ref + SCORE_ATOL), f"t {t}: score {err.max():.2e}"
                stats["score"] = max(stats["score"], float(np.max(err / np.maximum(ref, 1e-30))))
                un.S[:un.L] = np.where(np.arange(un.L) < wl.n_sink, 0, S[:un.L])
            g_route_run()
            torch.cuda.synchronize(dev)
            cache.qe_layer_info_sync()
            for un in units.values():
                un.rerank()
            for (b, layer, h), un in units.items():
                u = b * Hkv + h
                tiers = cache.token_tiers(layer)[u]
                assert np.array_equal(tiers[:un.L], un.tier[:un.L]), f"t {t} unit {(b, layer, h)}: tiers"
                quant = [p for p in range(un.L) if un.tier[p] in (H.INT4, H.INT2, H.NQ1)]
                for p in quant[::37]:
                    tier, _, _, kc, vc, par = cache.token(layer, u, p)
                    tc = un.codes[p]
                    assert tier == tc.tier and np.array_equal(kc, tc.k_codes) and np.array_equal(vc, tc.v_codes)
                    ref_par = np.array([tc.k_p0, tc.k_p1, tc.v_p0, tc.v_p1], np.float32)
                    assert np.array_equal(par.view(np.uint32), ref_par.view(np.uint32))
                    stats["codes"] += 1
    cache.qe_synchronize()
    print(f"hqe_16k: max out rel-L2 {stats['out']:.2e}, max score rel {stats['score']:.2e}, codes {stats['codes']}, "
          f"counts layer 0 unit 0 {cache.token_counts(0)[0].tolist()}")
    assert stats["codes"] > 0


def _adversarial_bf16_rows(D, rng):
    """bf16 rows whose exact mean and std stress the rebuild's 1-bit statistics: values 2^50
    below their neighbours (the wide path), magnitudes from 2^-60 to 2^8, bf16 subnormals,
    tiny normals, a constant row, cancelling pairs, one nonzero value, and a row whose exact
    mean 1 + 2^-24 lies halfway between two float32 values."""
    rows = []
    r = rng.standard_normal(D).astype(np.float32)
    r[::5] *= np.float32(2.0 ** -50)
    rows.append(r)
    rows.append(rng.standard_normal(D).astype(np.float32) * np.exp2(rng.integers(-60, 9, D)).astype(np.float32))
    rows.append((rng.integers(-120, 121, D) * 2.0 ** -133).astype(np.float32))   # subnormal bf16
    rows.append((rng.standard_normal(D) * 1e-35).astype(np.float32))
    rows.append(np.full(D, 1.5, np.float32))
    r = rng.standard_normal(D).astype(np.float32) * 4
    r[D // 2:] = -r[:D // 2]
    r[1] = np.float32(r[1] * np.float32(1.0078125))
    rows.append(r)
    r = np.zeros(D, np.float32)
    r[7] = np.float32(-2.25)
    rows.append(r)
    r = np.ones(D, np.float32)
    r[0], r[1] = np.float32(2.0), np.float32(2.0 ** -17)
    r[2:] = 1.0
    r[-1] = 0.0
    rows.append(r)
    return gen.bf16_bits_rne(np.stack(rows))   # rounded to bf16 (most rows already are bf16 values)


class PlantedTokRun(TokRun):
    """A five-tier run whose prefill carries adversarial key and value rows at chosen positions."""

    def __init__(self, wl, plant):
        super().__init__(wl)
        self.plant = plant   # position -> (key bits [D], value bits [D])

    def prefill(self):
        wl = self.wl
        for layer in range(wl.n_layers):
            K, V = host_kv(wl, layer, 0, wl.prefill, wl.batch)
            for p, (kr, vr) in self.plant.items():
                K[:, :, p] = kr
                V[:, :, p] = vr
            self.cache.qe_append(layer, self.place(K), self.place(V), wl.prefill)
            self.cache.qe_synchronize()
            for b in range(wl.batch):
                for h in range(wl.n_kv_heads):
                    self.units[(b, layer, h)].append(gen.bf16_bits_to_f32(K[b, h]), gen.bf16_bits_to_f32(V[b, h]))


@pytest.mark.parametrize("D", [128, 64])
def test_five_tier_adversarial_rows_one_bit(D):
    """Adversarial rows reach the 1-bit tier through the rebuild kernel (90 % of the ranked tokens
    go 1-bit): their codes and float32 mean and std equal the oracle's exact values rounded once,
    bit for bit, and attention over them follows the oracle."""
    G = 4 if D == 128 else 2
    wl = dataclasses.replace(BASE, name=f"adversarial_d{D}", head_dim=D, n_q_heads=2 * G, n_kv_heads=2, batch=1,
                             n_layers=1, prefill=300, decode_steps=16, route_period=16, score_window=0, n_sink=4,
                             n_recent=16, frac_bf16=0.1, frac_int4=0.0, frac_int2=0.0, frac_nq1=0.9, seed=77 + D)
    rng = np.random.default_rng(D)
    krows, vrows = _adversarial_bf16_rows(D, rng), _adversarial_bf16_rows(D, rng)[::-1]
    plant = {}
    for i in range(3 * len(krows)):                  # each row three times, at spread positions
        plant[30 + 9 * i] = (krows[i % len(krows)], vrows[(i + 1) % len(vrows)])
    run = PlantedTokRun(wl, plant)
    run.prefill()
    for _ in range(wl.decode_steps):
        run.step()
    run.cache.qe_synchronize()
    one_bit = sum(int(run.units[(0, 0, h)].tier[p] == H.NQ1) for h in range(wl.n_kv_heads) for p in plant)
    print(f"adversarial d{D}: planted tokens in the 1-bit tier {one_bit} of {2 * len(plant)}, "
          f"codes compared {run.codes_checked}, max out rel-L2 {run.max_out:.2e}")
    assert run.codes_checked > 0 and one_bit >= len(plant)
