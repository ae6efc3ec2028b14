"""qe_decode_step_noalloc (GPU): the decode step for callers that may not allocate device
memory gives the same outputs as qe_decode_step.

Two caches are built identically; at each of two steps in a row, one runs qe_decode_step and
the other the no-allocation entry point on the same inputs, and the outputs must agree within
the parity tolerance the other tests use.  This file is collected last on purpose."""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from qe_testlib import OUT_TOL, host_kv, host_q, torch_dev

pytestmark = pytest.mark.gpu

WL = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="noalloc", batch=2, n_q_heads=8, n_kv_heads=2,
                         head_dim=128, prefill=32 * 12 + 9, decode_steps=16, window=32, route_period=8, n_sink=5,
                         n_recent=32, kf=3, kq=4, plant_tokens=(), seed=41)


def _cache(stream):
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    c = qe.QECache(qe.config_from_workload(WL), stream.cuda_stream)
    K, V = host_kv(WL, 0, 0, WL.prefill, WL.batch)
    c.qe_append(0, torch.from_numpy(K.view(np.int16)).to(dev), torch.from_numpy(V.view(np.int16)).to(dev), WL.prefill)
    return c


def test_noalloc_matches_decode_step_two_calls():
    torch, dev = torch_dev()
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    a, b = _cache(stream), _cache(stream)
    out_a = torch.empty(WL.batch, WL.n_q_heads, WL.head_dim, device=dev, dtype=torch.float32)
    out_b = torch.empty_like(out_a)
    # reach a state with 2-bit windows: one routing event on both caches
    for t in range(1, WL.route_period + 3):
        K, V = host_kv(WL, 0, WL.prefill + t - 1, 1, WL.batch)
        k = torch.from_numpy(K.view(np.int16)).to(dev)
        v = torch.from_numpy(V.view(np.int16)).to(dev)
        q = torch.from_numpy(host_q(WL, 0, t, WL.batch).view(np.int16)).to(dev)
        a.qe_append(0, k, v, 1)
        b.qe_append(0, k, v, 1)
        if t <= WL.route_period:
            a.qe_decode_step(0, q, out_a)
            b.qe_decode_step(0, q, out_b)
            if t == WL.route_period:
                a.qe_route(0)
                b.qe_route(0)
            continue
        # two calls in a row of the no-allocation entry point against qe_decode_step
        a.qe_decode_step(0, q, out_a)
        b.qe_decode_step_noalloc(0, q, out_b)
        torch.cuda.synchronize()
        ga, gb = out_a.cpu().numpy(), out_b.cpu().numpy()
        for bb in range(WL.batch):
            for h in range(WL.n_q_heads):
                err = np.linalg.norm(gb[bb, h] - ga[bb, h]) / np.linalg.norm(ga[bb, h])
                assert err <= OUT_TOL, (t, bb, h, err)
    a.qe_synchronize()
    b.qe_synchronize()
    # the scores the two entry points accumulated agree too
    sa, sb = a.scores(0), b.scores(0)
    assert np.allclose(sa, sb, rtol=1e-4, atol=1e-7)
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
