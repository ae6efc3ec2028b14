"""Helpers shared by the GPU parity tests: drive the CUDA path through the C ABI and the CPU
oracle side by side on the same seeded inputs and compare.

Comparison protocol
-------------------
* attention outputs: relative L2 error per (batch, query head) <= 2e-3 against the fp64 oracle;
* accumulated window scores: |S_gpu - S_oracle| <= 1e-4 * S_oracle + 1e-7;
* 2-bit codes: identical; float32 min/scale: bitwise identical;
* tiers: identical at every routing event, unless the oracle's cutoff margin (lowest kept
  score minus highest dropped score, H2O page §5.1) at a changed cut is below 1e-4 relative:
  then both branches are correct, the two runs diverge and the unit is no longer compared.
  Such a unit is recorded with its margin; every test then calls ``assert_all_live``, so a run
  in which any compared unit stopped being compared fails (none of the seeded cases has a cut
  that close).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

import qe_inputs as gen
from oracle.quant import QuantizedWindow
from oracle.router import EVICTED, FULL, PINNED, QUANT
from oracle.run import make_unit

TIER_CODE = {PINNED: 1, FULL: 2, QUANT: 3, EVICTED: 4}
OUT_TOL = 2e-3
SCORE_RTOL = 1e-4
SCORE_ATOL = 1e-7
MARGIN_RTOL = 1e-4


def torch_dev():
    import torch
    return torch, torch.device("cuda:0")


def host_kv(wl, layer: int, pos0: int, n: int, batch: int):
    """[B][H_kv][n][d] uint16 bf16 bits of K and V from the CPU generator."""
    d = wl.head_dim
    K = np.zeros((batch, wl.n_kv_heads, n, d), np.uint16)
    V = np.zeros_like(K)
    for b in range(batch):
        for h in range(wl.n_kv_heads):
            K[b, h], V[b, h] = gen.gen_keys_values(wl, b, layer, h, pos0, n)
    return K, V


def host_q(wl, layer: int, step: int, batch: int):
    Q = np.zeros((batch, wl.n_q_heads, wl.head_dim), np.uint16)
    for b in range(batch):
        Q[b] = gen.gen_queries(wl, b, layer, range(wl.n_q_heads), step)
    return Q


def to_dev(a: np.ndarray):
    torch, dev = torch_dev()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


@dataclasses.dataclass
class Tracked:
    b: int
    layer: int
    kvh: int
    unit: object
    live: bool = True
    note: str = ""


class ParityRun:
    """A cache on the GPU plus oracle units for a chosen set of (b, layer, kvh)."""

    def __init__(self, wl, batch: int, n_layers: int, track: Sequence[Tuple[int, int, int]],
                 device_inputs: bool = False, host: Optional[str] = None, out_fp32: bool = True):
        """host: None (device buffers), "pinned" (page-locked torch tensors) or "pageable"
        (numpy arrays): where the inputs and the outputs of every call live.  out_fp32: the
        cache's output type (float32, else bf16; outputs are read back as float32)."""
        import tiered_quantize_evict_gb300 as qe
        torch, dev = torch_dev()
        self.torch, self.dev = torch, dev
        self.wl, self.batch, self.n_layers = wl, batch, n_layers
        self.cache = qe.QECache(qe.config_from_workload(wl, batch=batch, n_layers=n_layers, out_fp32=out_fp32),
                                torch.cuda.current_stream().cuda_stream)
        self.out_fp32 = out_fp32
        self.units_per_layer = batch * wl.n_kv_heads
        self.tracked = [Tracked(b, l, h, make_unit(wl)) for (b, l, h) in track]
        self.device_inputs = device_inputs
        self.gdev = None
        if device_inputs:
            import qe_inputs.cuda as gc
            gwl = dataclasses.replace(wl, batch=batch)
            self.gdev = gc.DeviceGenerator(gwl)
        self.t = 0
        self.max_out_err = 0.0
        self.max_score_err = 0.0
        self.ambiguous = 0
        self.codes_checked = 0
        self.route_events = 0
        assert host in (None, "pinned", "pageable") and not (host and device_inputs)
        self.host = host
        self.out = self.out_buffer((batch, wl.n_q_heads, wl.head_dim))

    def out_buffer(self, shape):
        """An output buffer of the cache's output type, where this run keeps its buffers."""
        torch = self.torch
        tdt = torch.float32 if self.out_fp32 else torch.bfloat16
        if self.host == "pinned":
            return torch.empty(*shape, dtype=tdt).pin_memory()
        if self.host == "pageable":
            return np.zeros(shape, np.float32 if self.out_fp32 else np.uint16)
        return torch.empty(*shape, device=self.dev, dtype=tdt)

    def read_buffer(self, out) -> np.ndarray:
        """An output buffer's values as float32 (the stream has passed the call)."""
        if isinstance(out, np.ndarray):
            a = np.array(out, copy=True)
            return a if self.out_fp32 else gen.bf16_bits_to_f32(a)
        return out.float().cpu().numpy().copy()

    def _place(self, a: np.ndarray):
        a = np.ascontiguousarray(a).view(np.int16)
        if self.host == "pinned":
            return self.torch.from_numpy(a).pin_memory()
        if self.host == "pageable":
            return a.copy()
        return to_dev(a)

    def _read_out(self):
        if self.host:   # host buffers are complete once the stream has passed the call
            self.cache.qe_synchronize()
        return self.read_buffer(self.out)

    # ------------------------------------------------------------------ inputs
    def _kv(self, layer, pos0, n):
        torch = self.torch
        if self.gdev is not None:
            k = torch.empty(self.batch, self.wl.n_kv_heads, n, self.wl.head_dim, device=self.dev, dtype=torch.int16)
            v = torch.empty_like(k)
            self.gdev.keys_values(layer, pos0, n, k, v, torch.cuda.current_stream().cuda_stream)
            return k, v
        K, V = host_kv(self.wl, layer, pos0, n, self.batch)
        return self._place(K), self._place(V)

    def _q(self, layer, step):
        torch = self.torch
        if self.gdev is not None:
            q = torch.empty(self.batch, self.wl.n_q_heads, self.wl.head_dim, device=self.dev, dtype=torch.int16)
            self.gdev.queries(layer, step, q, torch.cuda.current_stream().cuda_stream)
            return q
        return self._place(host_q(self.wl, layer, step, self.batch))

    # ------------------------------------------------------------------ driving
    def prefill(self):
        wl = self.wl
        for layer in range(self.n_layers):
            k, v = self._kv(layer, 0, wl.prefill)
            self.cache.qe_append(layer, k, v, wl.prefill)
            if self.host:   # the copies read host memory in stream order
                self.cache.qe_synchronize()
            del k, v
        for tr in self.tracked:
            kb, vb = gen.gen_keys_values(wl, tr.b, tr.layer, tr.kvh, 0, wl.prefill)
            tr.unit.append(gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb))

    def step(self, check: bool = True):
        """One decode step of every layer; compares the tracked units."""
        wl = self.wl
        self.t += 1
        t = self.t
        pos = wl.prefill + t - 1
        outs = {}
        for layer in range(self.n_layers):
            k, v = self._kv(layer, pos, 1)
            self.cache.qe_append(layer, k, v, 1)
            q = self._q(layer, t)
            self.cache.qe_decode_step(layer, q, self.out)
            if self.host or any(tr.layer == layer and tr.live for tr in self.tracked):
                # host inputs stay referenced (and unchanged) until the stream has read them
                outs[layer] = self._read_out()
        for tr in self.tracked:
            if not tr.live:
                continue
            heads = range(tr.kvh * wl.group, (tr.kvh + 1) * wl.group)
            q = gen.bf16_bits_to_f32(gen.gen_queries(wl, tr.b, tr.layer, heads, t))
            kb, vb = gen.gen_keys_values(wl, tr.b, tr.layer, tr.kvh, pos, 1)
            o_ref, _, _ = tr.unit.decode_step(q, gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb))
            if check:
                got = outs[tr.layer][tr.b, tr.kvh * wl.group:(tr.kvh + 1) * wl.group].astype(np.float64)
                for i in range(wl.group):
                    err = np.linalg.norm(got[i] - o_ref[i]) / np.linalg.norm(o_ref[i])
                    self.max_out_err = max(self.max_out_err, err)
                    assert err <= OUT_TOL, (f"step {t} unit {(tr.b, tr.layer, tr.kvh)} head {i}: "
                                            f"output rel-L2 {err:.3e} > {OUT_TOL}")
        if t % wl.route_period == 0:
            self.route_and_check()

    def check_scores(self):
        wl = self.wl
        by_layer = {}
        for tr in self.tracked:
            if not tr.live:
                continue
            if tr.layer not in by_layer:
                by_layer[tr.layer] = self.cache.scores(tr.layer)
            u = tr.b * wl.n_kv_heads + tr.kvh
            gs = by_layer[tr.layer][u]
            for j, s_ref in tr.unit.S.items():
                if tr.unit.tier[j] == EVICTED:
                    continue
                s_ref = float(s_ref)
                err = abs(float(gs[j]) - s_ref)
                self.max_score_err = max(self.max_score_err, err / max(s_ref, 1e-30))
                assert err <= SCORE_RTOL * s_ref + SCORE_ATOL, (
                    f"step {self.t} unit {(tr.b, tr.layer, tr.kvh)} window {j}: score {gs[j]} vs {s_ref}")

    def route_and_check(self, gpu_routed: bool = False):
        """Route the oracle units (and the cache, unless a replayed graph already did) and
        compare tiers and codes; scores are compared first (routing leaves them unchanged)."""
        wl = self.wl
        self.check_scores()
        if not gpu_routed:
            self.cache.qe_route(-1)
        self.route_events += 1
        tiers = {}
        for tr in self.tracked:
            if not tr.live:
                continue
            res = tr.unit.route()
            if tr.layer not in tiers:
                tiers[tr.layer] = self.cache.tiers(tr.layer)
            u = tr.b * wl.n_kv_heads + tr.kvh
            got = tiers[tr.layer][u]
            mism = [j for j, z in tr.unit.tier.items() if got[j] != TIER_CODE[z]]
            if mism:
                def rel(m, i):
                    if not (0 < i < len(res.order)):
                        return float("inf")
                    s = float(tr.unit.S[res.order[i - 1]])
                    return m / max(s, 1e-30)
                amb = min(rel(res.margin_f, res.kf), rel(res.margin_q, res.kf + res.kq))
                assert amb <= MARGIN_RTOL, (
                    f"step {self.t} unit {(tr.b, tr.layer, tr.kvh)}: tiers differ at windows {mism[:8]} "
                    f"(gpu {[int(got[j]) for j in mism[:8]]}, oracle {[tr.unit.tier[j] for j in mism[:8]]}) "
                    f"with margin {amb:.2e}")
                tr.live = False
                tr.note = f"tie-ambiguous at step {self.t} (margin {amb:.1e})"
                self.ambiguous += 1
                continue
            self.check_codes(tr)

    def assert_all_live(self):
        """Every tracked unit was compared to the end (no tie-ambiguous routing event)."""
        dropped = [(tr.b, tr.layer, tr.kvh, tr.note) for tr in self.tracked if not tr.live]
        assert not dropped and self.ambiguous == 0, f"units no longer compared: {dropped}"

    def check_codes(self, tr: Tracked, windows: Optional[List[int]] = None):
        wl = self.wl
        u = tr.b * wl.n_kv_heads + tr.kvh
        for j, z in tr.unit.tier.items():
            if z != QUANT or (windows is not None and j not in windows):
                continue
            q: QuantizedWindow = tr.unit.ledger[j]
            kc, vc, kz, ks, vz, vs = self.cache.quant_window(tr.layer, u, j)
            lo = wl.n_sink if j == 0 else 0
            assert np.array_equal(kc[lo:], q.k_codes), f"window {j}: key codes differ"
            assert np.array_equal(vc[lo:], q.v_codes), f"window {j}: value codes differ"
            assert np.array_equal(kz.view(np.uint32), q.k_min.view(np.uint32)), f"window {j}: key min differs"
            assert np.array_equal(ks.view(np.uint32), q.k_scale.view(np.uint32)), f"window {j}: key scale differs"
            assert np.array_equal(vz[lo:].view(np.uint32), q.v_min[:, 0].view(np.uint32)), f"window {j}: value min"
            assert np.array_equal(vs[lo:].view(np.uint32), q.v_scale[:, 0].view(np.uint32)), f"window {j}: value scale"
            self.codes_checked += 1

    def check_bf16_windows(self, tr: Tracked):
        """Full windows hold exactly the original bf16 values (promotion restores them)."""
        wl = self.wl
        u = tr.b * wl.n_kv_heads + tr.kvh
        n = 0
        for j, z in tr.unit.tier.items():
            if z != FULL:
                continue
            k, v = self.cache.bf16_window(tr.layer, u, j)
            lo, hi = tr.unit.window_range(j)
            kk = gen.bf16_bits_to_f32(k[lo - j * wl.window:hi - j * wl.window])
            vv = gen.bf16_bits_to_f32(v[lo - j * wl.window:hi - j * wl.window])
            assert np.array_equal(kk, tr.unit.K[lo:hi]) and np.array_equal(vv, tr.unit.V[lo:hi]), f"window {j}"
            n += 1
        return n
