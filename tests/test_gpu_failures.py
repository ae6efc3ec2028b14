"""Failure paths (GPU), exercised without faulting the GPU (H2O page §5.1: canaries and a
fallback; the library reports failures as status codes).

- A bounded device wait that expires: qe_debug_inject(QE_DEBUG_EXPIRE_WAIT) makes every warp of
  one decode step's attention report a wait as expired once the tile's copy has landed (so no
  copy is in flight when a CTA leaves).  qe_synchronize must return QE_ERR_TIMEOUT, and the GPU
  must stay usable: a new cache on it follows the oracle.  Both tierings.
- A device allocation that fails inside qe_init, at every allocation site in turn: QE_ERR_OOM
  naming the buffer, nothing leaked, the next qe_init succeeds.
- A pinned host backing store that cannot be allocated: QE_ERR_HOST_STORE.
"""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
from qe_testlib import OUT_TOL, ParityRun, torch_dev

pytestmark = pytest.mark.gpu

WL = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="failures", batch=2, n_q_heads=8, n_kv_heads=2,
                         head_dim=128, prefill=32 * 10 + 3, decode_steps=12, window=32, route_period=4, n_sink=5,
                         n_recent=32, kf=3, kq=4, plant_tokens=(), seed=61)
HQE = dataclasses.replace(gen.WORKLOADS["tiny_hqe"], name="failures_hqe", n_layers=1, decode_steps=12,
                          route_period=6, score_window=3)


def _follow(wl, steps):
    """A fresh cache on the same GPU, every unit against the oracle for `steps` steps."""
    track = [(b, 0, h) for b in range(wl.batch) for h in range(wl.n_kv_heads)]
    run = ParityRun(dataclasses.replace(wl, n_layers=1), wl.batch, 1, track)
    run.prefill()
    for _ in range(steps):
        run.step()
    run.cache.qe_synchronize()
    run.assert_all_live()
    run.cache.close()
    return run.max_out_err


@pytest.mark.parametrize("kind", ["windows", "tokens"])
def test_expired_wait_reports_timeout_and_the_gpu_stays_usable(kind):
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    wl = WL if kind == "windows" else HQE
    c = qe.QECache(qe.config_from_workload(wl, n_layers=1))
    B, Hkv, Hq, D = wl.batch, wl.n_kv_heads, wl.n_q_heads, wl.head_dim
    K = torch.zeros(B, Hkv, wl.prefill, D, device=dev, dtype=torch.int16)
    c.qe_append(0, K, K, wl.prefill)
    k1 = torch.zeros(B, Hkv, 1, D, device=dev, dtype=torch.int16)
    q = torch.zeros(B, Hq, D, device=dev, dtype=torch.int16)
    out = torch.empty(B, Hq, D, device=dev, dtype=torch.float32)
    for _ in range(2):
        c.qe_append(0, k1, k1, 1)
        c.qe_decode_step(0, q, out)
    c.qe_synchronize()                                   # healthy so far
    assert qe.debug_inject(qe.QE_DEBUG_EXPIRE_WAIT, 1, c) == qe.QE_OK
    c.qe_append(0, k1, k1, 1)
    c.qe_decode_step(0, q, out)
    with pytest.raises(qe.QEError) as e:
        c.qe_synchronize()
    assert e.value.status == qe.QE_ERR_TIMEOUT, str(e.value)
    with pytest.raises(qe.QEError):                      # the flag is sticky
        c.qe_synchronize()
    c.close()
    torch.cuda.synchronize(dev)                          # the context is intact
    assert _follow(WL, 6) <= OUT_TOL


@pytest.mark.parametrize("kind", ["windows", "tokens"])
def test_every_device_allocation_failure_is_reported(kind):
    import tiered_quantize_evict_gb300 as qe
    torch, dev = torch_dev()
    wl = WL if kind == "windows" else HQE
    cfg = qe.config_from_workload(wl, n_layers=1)
    torch.cuda.synchronize(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    failed = 0
    for n in range(1, 200):
        assert qe.debug_inject(qe.QE_DEBUG_FAIL_DEVICE_ALLOC, n) == qe.QE_OK
        try:
            c = qe.QECache(cfg)
        except qe.QEError as err:
            assert err.status == qe.QE_ERR_OOM and "injected" in str(err), (n, str(err))
            failed += 1
            continue
        # n passed the number of allocations: qe_init succeeded and the injection never fired
        qe.debug_inject(qe.QE_DEBUG_FAIL_DEVICE_ALLOC, 0)
        c.close()
        break
    else:
        raise AssertionError("qe_init never succeeded")
    assert failed >= 10, failed                         # every allocation site was hit once
    torch.cuda.synchronize(dev)
    free1 = torch.cuda.mem_get_info(dev)[0]
    assert free0 - free1 < (64 << 20), (free0, free1)   # nothing of note leaked
    assert _follow(WL, 4) <= OUT_TOL


def test_host_store_failure_is_reported():
    import tiered_quantize_evict_gb300 as qe
    cfg = qe.config_from_workload(WL, n_layers=1)
    assert qe.debug_inject(qe.QE_DEBUG_FAIL_HOST_STORE, 1) == qe.QE_OK
    with pytest.raises(qe.QEError) as e:
        qe.QECache(cfg)
    assert e.value.status == qe.QE_ERR_HOST_STORE, str(e.value)
    c = qe.QECache(cfg)                                  # one-shot: the next init succeeds
    c.close()
