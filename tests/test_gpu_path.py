"""Parity of the CUDA path with the CPU oracle through the C ABI (GPU)."""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from qe_testlib import ParityRun, host_kv, host_q, to_dev, torch_dev

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host_generator():
    import qe_inputs.cuda as gc
    torch, dev = torch_dev()
    wl = dataclasses.replace(gen.WORKLOADS["throughput_32k"], batch=2)
    g = gc.DeviceGenerator(wl)
    k = torch.empty(2, wl.n_kv_heads, 40, wl.head_dim, device=dev, dtype=torch.int16)
    v = torch.empty_like(k)
    g.keys_values(3, 1000, 40, k, v)
    K, V = host_kv(wl, 3, 1000, 40, 2)
    assert np.array_equal(k.cpu().numpy().view(np.uint16), K)
    assert np.array_equal(v.cpu().numpy().view(np.uint16), V)
    for step in (1, 64, 65, 128):
        q = torch.empty(2, wl.n_q_heads, wl.head_dim, device=dev, dtype=torch.int16)
        g.queries(5, step, q)
        assert np.array_equal(q.cpu().numpy().view(np.uint16), host_q(wl, 5, step, 2)), step


def test_tiny_workload_trajectory():
    """The 1-layer workload end to end: every output, score, tier and code at every step."""
    wl = gen.WORKLOADS["tiny_qevict"]
    run = ParityRun(wl, 1, 1, [(0, 0, 0)])
    run.prefill()
    for _ in range(wl.decode_steps):
        run.step()
    run.check_scores()
    run.cache.qe_synchronize()
    tr = run.tracked[0]
    assert tr.live, tr.note
    assert run.codes_checked > 0
    assert run.check_bf16_windows(tr) > 0
    st = run.cache.route_stats(0)
    assert st.routes == wl.decode_steps // wl.route_period
    # the planted window 4 was demoted and came back (it is Full at the end)
    assert st.promotions >= 1
    print(f"max out err {run.max_out_err:.2e}, max score rel err {run.max_score_err:.2e}")


def test_error_codes():
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    wl = gen.WORKLOADS["tiny_qevict"]
    c = qe.QECache(qe.config_from_workload(wl, max_context=40))
    q = torch.zeros(1, 4, 64, device=dev, dtype=torch.int16)
    out = torch.zeros(1, 4, 64, device=dev, dtype=torch.float32)
    with pytest.raises(qe.QEError) as e:
        c.qe_decode_step(0, q, out)
    assert e.value.status == qe.QE_ERR_STATE
    k = torch.zeros(1, 1, 41, 64, device=dev, dtype=torch.int16)
    with pytest.raises(qe.QEError) as e:
        c.qe_append(0, k, k, 41)
    assert e.value.status == qe.QE_ERR_CAPACITY
    with pytest.raises(qe.QEError) as e:
        c.qe_append(1, k, k, 1)
    assert e.value.status == qe.QE_ERR_INVALID_ARG
    c.qe_append(0, k[:, :, :20], k[:, :, :20], 20)
    with pytest.raises(qe.QEError) as e:
        c.quant_window(0, 0, 0)
    assert e.value.status == qe.QE_ERR_STATE
    c.qe_synchronize()
    c.close()


def test_launch_overhead_measure():
    """qe_launch_overhead times empty launches of the attention launch's shape: a positive
    number of microseconds well below a real attention launch, with the handle's state
    untouched; it refuses a bad count."""
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    wl = gen.WORKLOADS["tiny_qevict"]
    c = qe.QECache(qe.config_from_workload(wl, max_context=64))
    k = torch.zeros(1, 1, 20, 64, device=dev, dtype=torch.int16)
    c.qe_append(0, k, k, 20)
    before = c.layer_info(0).length
    us = c.launch_overhead(20)
    assert 0.0 < us < 50.0
    assert c.layer_info(0).length == before
    with pytest.raises(qe.QEError) as e:
        c.launch_overhead(0)
    assert e.value.status == qe.QE_ERR_INVALID_ARG
    c.qe_synchronize()
    c.close()
