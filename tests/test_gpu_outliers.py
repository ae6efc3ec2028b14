"""Attention over 2-bit windows holding outlier and tiny magnitudes (GPU), against the oracle.

QEvict notes §1 and KV-cache evolution §5: keys are quantized per channel because some key
channels carry outliers far larger than the rest.  The 2-bit tiles meet the tensor cores as f16
(q s_K for keys, 4 p s_V for values) unless a slot's recorded parameter magnitudes say the
products could leave the f16 range; such tiles take bf16 operands (keys as three exact bf16
parts).  Keys stored pre-RoPE always meet the query as three exact bf16 parts.

Inputs are seeded arrays, rounded to bf16:
- keys N(0,1) with a channel pair scaled by 10^3 (the query's same pair by 10^-3, so the logits
  stay moderate; pairs, because a rotation mixes the channels of a pair) and a pair scaled by
  10^-6;
- one window of tokens (keys and values) scaled by 10^-6;
- "moderate": value outliers scaled by 10; the 10^3 key channel stays on the f16 path and only
  the tiny window goes to bf16;
- "extreme": more key pairs scaled by 2 10^4 and 10^-6 with inverse query factors (a query
  pair of 10^6), value outliers scaled by 100 (4 p s_V past the f16 range) and by 10^-6:
  every 2-bit tile takes bf16 operands; the same data with keys stored pre-RoPE.

Every unit follows the oracle: outputs every step within 2e-3 relative L2, scores at every
routing event within 1e-4, tiers, 2-bit codes and float32 parameters bit for bit.
"""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from qe_testlib import OUT_TOL, ParityRun, to_dev

pytestmark = pytest.mark.gpu

BASE = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="outliers", batch=2, n_q_heads=8, n_kv_heads=2,
                           head_dim=128, prefill=32 * 14 + 7, decode_steps=24, window=32, route_period=8, n_sink=5,
                           n_recent=32, kf=4, kq=6, plant_tokens=(), outlier_mode="fixed", outlier_fixed=(), seed=91)


def _arrays(wl, extreme: bool, seed: int):
    rng = np.random.default_rng(seed)
    B, Hkv, Hq, D = wl.batch, wl.n_kv_heads, wl.n_q_heads, wl.head_dim
    Lt, T = wl.prefill + wl.decode_steps, wl.decode_steps
    K = rng.standard_normal((B, Hkv, Lt, D))
    V = rng.standard_normal((B, Hkv, Lt, D))
    Q = rng.standard_normal((T, B, Hq, D))
    # scales act on whole rotary pairs (2i, 2i + 1), which a rotation mixes
    K[..., 76:78] *= 1e-6                    # a tiny key pair (tiny per-channel scales)
    scales = {2: 1e3}
    if extreme:
        scales.update({16: 2e4, 40: 1e-6})   # query pair 40, 41 at 10^6
    for c, a in scales.items():
        K[..., c:c + 2] *= a
        Q[..., c:c + 2] /= a
    win = 6                                  # one window of tiny tokens
    K[:, :, win * wl.window:(win + 1) * wl.window] *= 1e-6
    V[:, :, win * wl.window:(win + 1) * wl.window] *= 1e-6
    pos = np.arange(Lt)
    V[:, :, (pos % 11) == 3] *= 100.0 if extreme else 10.0   # value outliers
    if extreme:
        V[:, :, (pos % 13) == 5] *= 1e-6
    bits = lambda a: gen.bf16_bits_rne(a.astype(np.float32))
    return bits(K), bits(V), bits(Q)


class ArrayRun(ParityRun):
    """ParityRun fed from explicit bf16 arrays instead of the workload generator."""

    def __init__(self, wl, K, V, Q):
        track = [(b, 0, h) for b in range(wl.batch) for h in range(wl.n_kv_heads)]
        super().__init__(wl, wl.batch, 1, track)
        self.K, self.V, self.Q = K, V, Q

    def prefill(self):
        L0 = self.wl.prefill
        self.cache.qe_append(0, to_dev(self.K[:, :, :L0]), to_dev(self.V[:, :, :L0]), L0)
        for tr in self.tracked:
            tr.unit.append(gen.bf16_bits_to_f32(self.K[tr.b, tr.kvh, :L0]),
                           gen.bf16_bits_to_f32(self.V[tr.b, tr.kvh, :L0]))

    def step(self, check: bool = True):
        wl = self.wl
        self.t += 1
        t, pos = self.t, wl.prefill + self.t - 1
        # a single-token append keeps its K and V pointers until the decode step's attention
        # launch writes the token: the buffers stay referenced until the output is read
        k, v = to_dev(self.K[:, :, pos:pos + 1]), to_dev(self.V[:, :, pos:pos + 1])
        self.cache.qe_append(0, k, v, 1)
        q = to_dev(self.Q[t - 1])
        self.cache.qe_decode_step(0, q, self.out)
        got = self._read_out()
        del k, v, q
        for tr in self.tracked:
            G = wl.group
            qh = gen.bf16_bits_to_f32(self.Q[t - 1, tr.b, tr.kvh * G:(tr.kvh + 1) * G])
            o, _, _ = tr.unit.decode_step(qh, gen.bf16_bits_to_f32(self.K[tr.b, tr.kvh, pos:pos + 1]),
                                          gen.bf16_bits_to_f32(self.V[tr.b, tr.kvh, pos:pos + 1]))
            for i in range(G):
                g_ = got[tr.b, tr.kvh * G + i].astype(np.float64)
                err = np.linalg.norm(g_ - o[i]) / np.linalg.norm(o[i])
                self.max_out_err = max(self.max_out_err, err)
                assert np.isfinite(g_).all() and err <= OUT_TOL, \
                    f"step {t} unit {(tr.b, tr.kvh)} head {i}: rel-L2 {err:.3e}"
        if t % wl.route_period == 0:
            self.route_and_check()


CASES = {
    "moderate": dict(extreme=False, rope=0.0),
    "extreme": dict(extreme=True, rope=0.0),
    "pre_rope_extreme": dict(extreme=True, rope=10000.0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_outlier_magnitudes_follow_the_oracle(name):
    c = CASES[name]
    wl = dataclasses.replace(BASE, name="outliers_" + name, rope_theta=c["rope"])
    K, V, Q = _arrays(wl, c["extreme"], seed=7 + len(name))
    run = ArrayRun(wl, K, V, Q)
    run.prefill()
    for _ in range(wl.decode_steps):
        run.step()
    run.check_scores()
    run.cache.qe_synchronize()
    run.assert_all_live()
    assert run.codes_checked > 0 and run.route_events == wl.decode_steps // wl.route_period
    for tr in run.tracked:
        run.check_bf16_windows(tr)
    # the tiny window and the value outliers sit in 2-bit windows at the end
    quant_windows = {j for tr in run.tracked for j, z in tr.unit.tier.items() if z == "Q"}
    print(f"{name}: max out rel-L2 {run.max_out_err:.2e}, max score rel {run.max_score_err:.2e}, "
          f"2-bit windows compared {run.codes_checked}, quantized windows {sorted(quant_windows)}")
    assert quant_windows
