"""qe_decode_step_noalloc (GPU): the decode step for callers that may not allocate device
memory gives the same outputs as qe_decode_step, and both follow the oracle.

Two caches are built identically; at each of two steps in a row, one runs qe_decode_step and
the other the no-allocation entry point on the same inputs.  The outputs must agree with each
other and with the oracle's fp64 attention within the parity tolerance the other tests use, and
the window scores both accumulated must match the oracle's.  Small cases check the refusals:
a layer awaiting qe_verify_commit, too many units, too many tiles.  This file is collected last
on purpose."""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from oracle.router import EVICTED
from oracle.run import make_unit
from qe_testlib import OUT_TOL, SCORE_ATOL, SCORE_RTOL, host_kv, host_q, torch_dev

pytestmark = pytest.mark.gpu

WL = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="noalloc", batch=2, n_q_heads=8, n_kv_heads=2,
                         head_dim=128, prefill=32 * 12 + 9, decode_steps=16, window=32, route_period=8, n_sink=5,
                         n_recent=32, kf=3, kq=4, plant_tokens=(), seed=41)


def _cache(stream, wl=WL):
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    c = qe.QECache(qe.config_from_workload(wl), stream.cuda_stream)
    K, V = host_kv(wl, 0, 0, wl.prefill, wl.batch)
    c.qe_append(0, torch.from_numpy(K.view(np.int16)).to(dev), torch.from_numpy(V.view(np.int16)).to(dev), wl.prefill)
    return c


def _oracle_units(wl):
    units = {}
    for b in range(wl.batch):
        for h in range(wl.n_kv_heads):
            u = make_unit(wl)
            kb, vb = gen.gen_keys_values(wl, b, 0, h, 0, wl.prefill)
            u.append(gen.bf16_bits_to_f32(kb), gen.bf16_bits_to_f32(vb))
            units[(b, h)] = u
    return units


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def test_noalloc_matches_decode_step_two_calls():
    torch, dev = torch_dev()
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    a, b = _cache(stream), _cache(stream)
    units = _oracle_units(WL)
    out_a = torch.empty(WL.batch, WL.n_q_heads, WL.head_dim, device=dev, dtype=torch.float32)
    out_b = torch.empty_like(out_a)
    G = WL.group
    noalloc_calls = 0
    # reach a state with 2-bit windows: one routing event on both caches and the oracle units
    for t in range(1, WL.route_period + 3):
        K, V = host_kv(WL, 0, WL.prefill + t - 1, 1, WL.batch)
        k = torch.from_numpy(K.view(np.int16)).to(dev)
        v = torch.from_numpy(V.view(np.int16)).to(dev)
        Q = host_q(WL, 0, t, WL.batch)
        q = torch.from_numpy(Q.view(np.int16)).to(dev)
        a.qe_append(0, k, v, 1)
        b.qe_append(0, k, v, 1)
        ref = {}
        for (bb, h), u in units.items():
            o, _, _ = u.decode_step(gen.bf16_bits_to_f32(Q[bb, h * G:(h + 1) * G]),
                                    gen.bf16_bits_to_f32(K[bb, h]), gen.bf16_bits_to_f32(V[bb, h]))
            ref[(bb, h)] = o
        if t <= WL.route_period:
            a.qe_decode_step(0, q, out_a)
            b.qe_decode_step(0, q, out_b)
            if t == WL.route_period:
                a.qe_route(0)
                b.qe_route(0)
                for u in units.values():
                    u.route()
            continue
        # two calls in a row of the no-allocation entry point against qe_decode_step and the oracle
        a.qe_decode_step(0, q, out_a)
        b.qe_decode_step_noalloc(0, q, out_b)
        noalloc_calls += 1
        torch.cuda.synchronize()
        ga, gb = out_a.cpu().numpy(), out_b.cpu().numpy()
        for bb in range(WL.batch):
            for h in range(WL.n_q_heads):
                o_ref = ref[(bb, h // G)][h % G]
                assert _rel(gb[bb, h], ga[bb, h]) <= OUT_TOL, (t, bb, h)
                assert _rel(gb[bb, h].astype(np.float64), o_ref) <= OUT_TOL, (t, bb, h, "noalloc vs oracle")
                assert _rel(ga[bb, h].astype(np.float64), o_ref) <= OUT_TOL, (t, bb, h, "decode step vs oracle")
    assert noalloc_calls == 2
    a.qe_synchronize()
    b.qe_synchronize()
    # the scores both entry points accumulated agree with each other and with the oracle's
    sa, sb = a.scores(0), b.scores(0)
    assert np.allclose(sa, sb, rtol=SCORE_RTOL, atol=SCORE_ATOL)
    for (bb, h), u in units.items():
        row = sb[bb * WL.n_kv_heads + h]
        for j, s_ref in u.S.items():
            if u.tier[j] == EVICTED:
                continue
            assert abs(float(row[j]) - float(s_ref)) <= SCORE_RTOL * float(s_ref) + SCORE_ATOL, (bb, h, j)
    assert b.layer_info(0).n_quant > 0
    a.close()
    b.close()
    torch.cuda.set_stream(torch.cuda.default_stream(dev))


def test_noalloc_rejects_too_many_units():
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    wl = dataclasses.replace(WL, batch=9)   # 18 units > 16
    c = qe.QECache(qe.config_from_workload(wl))
    K = torch.zeros(wl.batch, wl.n_kv_heads, 40, wl.head_dim, device=dev, dtype=torch.int16)
    c.qe_append(0, K, K, 40)
    q = torch.zeros(wl.batch, wl.n_q_heads, wl.head_dim, device=dev, dtype=torch.int16)
    out = torch.empty(wl.batch, wl.n_q_heads, wl.head_dim, device=dev, dtype=torch.float32)
    with pytest.raises(qe.QEError) as e:
        c.qe_decode_step_noalloc(0, q, out)
    assert e.value.status == qe.QE_ERR_CAPACITY and "16" in str(e.value)
    c.qe_synchronize()
    c.close()


def test_noalloc_rejects_too_many_tiles():
    """One unit whose bf16 windows hold more than 8192 tiles of 16 tokens (a 140,000-token
    prefill at w 64): refused before any launch; qe_decode_step still serves it."""
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    n = 140_000
    wl = dataclasses.replace(WL, batch=1, n_q_heads=4, n_kv_heads=1, window=64, prefill=n, decode_steps=64)
    c = qe.QECache(qe.config_from_workload(wl, max_context=n + 64))
    K = torch.zeros(1, 1, n, wl.head_dim, device=dev, dtype=torch.int16)
    c.qe_append(0, K, K, n)
    q = torch.zeros(1, 4, wl.head_dim, device=dev, dtype=torch.int16)
    out = torch.empty(1, 4, wl.head_dim, device=dev, dtype=torch.float32)
    with pytest.raises(qe.QEError) as e:
        c.qe_decode_step_noalloc(0, q, out)
    assert e.value.status == qe.QE_ERR_CAPACITY and "8192" in str(e.value)
    c.qe_decode_step(0, q, out)
    c.qe_synchronize()
    c.close()


def test_noalloc_rejects_a_layer_awaiting_commit():
    """A pending speculative verify: the no-allocation step refuses the layer (its scores would
    take the drafts' masses) until qe_verify_commit, then serves it again."""
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    c = _cache(stream)
    G, B, D = WL.group, WL.batch, WL.head_dim
    n_q = 2
    qv = torch.zeros(n_q, B, WL.n_q_heads, D, device=dev, dtype=torch.int16)
    kv = torch.zeros(n_q, B, WL.n_kv_heads, D, device=dev, dtype=torch.int16)
    outv = torch.empty(n_q, B, WL.n_q_heads, D, device=dev, dtype=torch.float32)
    c.qe_verify(0, qv, kv, kv, outv, n_q)
    q = torch.zeros(B, WL.n_q_heads, D, device=dev, dtype=torch.int16)
    out = torch.empty(B, WL.n_q_heads, D, device=dev, dtype=torch.float32)
    with pytest.raises(qe.QEError) as e:
        c.qe_decode_step_noalloc(0, q, out)
    assert e.value.status == qe.QE_ERR_STATE
    c.qe_verify_commit(0, 1)
    c.qe_decode_step_noalloc(0, q, out)
    c.qe_synchronize()
    assert np.isfinite(out.cpu().numpy()).all() and G == 4
    c.close()
    torch.cuda.set_stream(torch.cuda.default_stream(dev))
