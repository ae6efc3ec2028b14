"""Pins of the oracle's decode attention and score accumulation (no GPU).

Special cases that reduce to a library routine: with nothing quantized or
evicted the tiered attention is plain softmax attention, checked against
torch's scaled_dot_product_attention in float64; windows whose values sit
exactly on the quantization grid dequantize exactly, so attention over them
also equals plain attention; evicted windows simply drop out.
"""
import numpy as np
import pytest
import torch

from oracle.qevict import QEvictUnit
from oracle.router import EVICTED, FULL, QUANT

RNG = np.random.default_rng(11)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _sdpa(q, K, V):
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, :, None, :]      # [1, G, 1, d]
    Kt = torch.from_numpy(np.asarray(K, np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    Vt = torch.from_numpy(np.asarray(V, np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)
    return o[0, :, 0, :].numpy()


def _unit(w=16, n_sink=4, n_recent=16, d=64, G=4, kf=100, kq=0, max_ctx=512):
    return QEvictUnit(w, n_sink, n_recent, d, G, lambda L: (kf, kq), max_ctx)


def test_full_precision_equals_sdpa_and_mass_is_conserved():
    u = _unit()
    L0 = 200
    K = _bf16(RNG.standard_normal((L0 + 10, 64)))
    V = _bf16(RNG.standard_normal((L0 + 10, 64)))
    u.append(K[:L0], V[:L0])
    for t in range(10):
        q = _bf16(RNG.standard_normal((4, 64)))
        o, mass, sink = u.decode_step(q, K[L0 + t:L0 + t + 1], V[L0 + t:L0 + t + 1])
        ref = _sdpa(q, K[:L0 + t + 1], V[:L0 + t + 1])
        np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
        # per-window mass from an independent softmax: sum over heads, then over window tokens
        lg = torch.from_numpy(q.astype(np.float64)) @ torch.from_numpy(K[:L0 + t + 1].astype(np.float64)).T
        p = torch.softmax(lg / 8.0, dim=-1).sum(0).numpy()
        for j, m in mass.items():
            lo = 4 if j == 0 else 16 * j
            np.testing.assert_allclose(m, p[lo:min(16 * j + 16, L0 + t + 1)].sum(), rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(sink, p[:4].sum(), rtol=1e-12)
        assert abs(sum(mass.values()) + sink - 4.0) < 1e-12
        if t == 4:
            u.route()


def test_grid_valued_quantized_windows_equal_full_attention():
    """All routable windows go to INT2; their values lie on the grid, so nothing changes."""
    w, d, n_sink = 16, 64, 4
    L0 = 128
    u = _unit(w=w, n_sink=n_sink, n_recent=16, d=d, kf=0, kq=100)
    K = RNG.standard_normal((L0 + 1, d)).astype(np.float32)
    V = RNG.standard_normal((L0 + 1, d)).astype(np.float32)
    for j in range(L0 // w):
        rows = np.arange(j * w + (n_sink if j == 0 else 0), (j + 1) * w)
        ck = RNG.integers(0, 4, (len(rows), d))
        ck[0], ck[1] = 0, 3                       # each key channel spans levels 0..3
        kz = RNG.integers(-8, 8, d) * 0.25
        K[rows] = kz + ck * 0.5
        cv = RNG.integers(0, 4, (len(rows), d))
        cv[:, 0], cv[:, 1] = 0, 3                 # each value token spans levels 0..3
        vz = RNG.integers(-8, 8, (len(rows), 1)) * 0.25
        V[rows] = vz + cv * 0.125
    u.append(K[:L0], V[:L0])
    res = u.route()
    assert len(res.quant) == 7 and not res.full and not res.evicted
    q = _bf16(RNG.standard_normal((4, d)))
    o, mass, sink = u.decode_step(q, K[L0:L0 + 1], V[L0:L0 + 1])
    np.testing.assert_allclose(o, _sdpa(q, K[:L0 + 1], V[:L0 + 1]), rtol=1e-12, atol=1e-12)


def test_evicted_windows_are_absent():
    w, d = 16, 64
    u = _unit(kf=2, kq=1)
    L0 = 160
    K = _bf16(RNG.standard_normal((L0 + 1, d)))
    V = _bf16(RNG.standard_normal((L0 + 1, d)))
    u.append(K[:L0], V[:L0])
    for j in u.tier:
        u.S[j] = np.float32(j % 5)                  # deterministic ranking
    res = u.route()
    assert len(res.full) == 2 and len(res.quant) == 1 and res.evicted
    q = _bf16(RNG.standard_normal((4, d)))
    o, mass, sink = u.decode_step(q, K[L0:L0 + 1], V[L0:L0 + 1])
    keep = list(range(4))
    for j, z in sorted(u.tier.items()):
        if z != EVICTED:
            lo, hi = u.window_range(j)
            keep += list(range(lo, hi))
    kacc = K[keep].astype(np.float64)
    vacc = V[keep].astype(np.float64)
    jq = res.quant[0]
    kh, vh = u.dequantized(jq)
    lo, hi = u.window_range(jq)
    idx = [keep.index(p) for p in range(lo, hi)]
    kacc[idx], vacc[idx] = kh, vh
    np.testing.assert_allclose(o, _sdpa(q, kacc, vacc), rtol=1e-12, atol=1e-12)
    assert all(j not in mass for j in res.evicted)


def test_scores_accumulate_in_float32():
    u = _unit()
    L0 = 64
    K = _bf16(RNG.standard_normal((L0 + 20, 64)))
    V = _bf16(RNG.standard_normal((L0 + 20, 64)))
    u.append(K[:L0], V[:L0])
    ref = {}
    for t in range(20):
        q = _bf16(RNG.standard_normal((4, 64)))
        _, mass, _ = u.decode_step(q, K[L0 + t:L0 + t + 1], V[L0 + t:L0 + t + 1])
        for j, m in mass.items():
            ref[j] = np.float32(ref.get(j, np.float32(0)) + np.float32(m))
    for j in ref:
        assert u.S[j] == ref[j] and u.S[j].dtype == np.float32
