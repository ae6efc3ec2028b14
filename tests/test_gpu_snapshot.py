"""Session restore (H2O page §6: a cache resumes from its tiers, scores, boundaries and
positions, not from its K and V alone): qe_snapshot / qe_restore on the GPU.

A cache runs decode steps and routing events against the oracle; its snapshot is restored into
a second handle of the same configuration that has run steps of its own; both then run the same
steps.  The restored handle's outputs, scores and tiers equal the original's bit for bit, and
the original keeps following the oracle, so the restored one does too.  Error paths: another
configuration, a damaged header, a layer awaiting qe_verify_commit, a five-tier handle."""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
import tiered_quantize_evict_gb300 as qe
from qe_testlib import ParityRun, host_kv, host_q, to_dev

pytestmark = pytest.mark.gpu

WL = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="snapshot", batch=2, n_q_heads=8, n_kv_heads=2,
                         head_dim=128, prefill=290, decode_steps=80, window=32, route_period=12, n_sink=5,
                         n_recent=32, kf=4, kq=6, plant_tokens=(), seed=61)


def test_restored_handle_continues_bit_for_bit():
    import torch
    wl = WL
    track = [(b, 0, h) for b in range(wl.batch) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, 1, track)
    run.prefill()
    for _ in range(30):                 # two routing events before the snapshot
        run.step()
    snap = run.cache.snapshot()
    assert snap.nbytes > 0 and bytes(snap[:8]) == b"QESNAP01"

    other = qe.QECache(qe.config_from_workload(wl, batch=wl.batch, n_layers=1),
                       torch.cuda.current_stream().cuda_stream)
    # the second handle has state of its own, which the restore replaces entirely
    K, V = host_kv(wl, 0, 0, 100, wl.batch)
    other.qe_append(0, to_dev(K), to_dev(V), 100)
    out_b = torch.empty(wl.batch, wl.n_q_heads, wl.head_dim, device=run.dev, dtype=torch.float32)
    other.qe_decode_step(0, to_dev(host_q(wl, 0, 1, wl.batch)), out_b)
    other.qe_route(-1)
    other.restore(snap)
    assert other.layer_info(0).length == run.cache.layer_info(0).length
    assert np.array_equal(other.tiers(0), run.cache.tiers(0))
    assert np.array_equal(other.scores(0), run.cache.scores(0))

    for _ in range(40):                 # three more routing events
        run.step()
        t = run.t
        pos = wl.prefill + t - 1
        k, v = run._kv(0, pos, 1)
        q = run._q(0, t)
        other.qe_append(0, k, v, 1)
        other.qe_decode_step(0, q, out_b)
        if t % wl.route_period == 0:
            other.qe_route(-1)
        got_a = run._read_out()
        got_b = out_b.cpu().numpy()
        del k, v, q
        assert np.array_equal(got_a, got_b), f"step {t}: outputs differ"
    run.cache.qe_synchronize()
    other.qe_synchronize()
    assert np.array_equal(other.tiers(0), run.cache.tiers(0))
    assert np.array_equal(other.scores(0), run.cache.scores(0))
    assert other.layer_info(0).length == run.cache.layer_info(0).length
    # the windows' contents too: a 2-bit window and a bf16 window of every unit
    tiers = run.cache.tiers(0)
    for u in range(wl.batch * wl.n_kv_heads):
        for code in (2, 3):             # Full (bf16), Quantized (2-bit)
            js = np.nonzero(tiers[u] == code)[0]
            if len(js) == 0:
                continue
            j = int(js[0])
            if code == 2:
                a, b = run.cache.bf16_window(0, u, j), other.bf16_window(0, u, j)
            else:
                a, b = run.cache.quant_window(0, u, j), other.quant_window(0, u, j)
            for x, y in zip(a, b):
                assert np.array_equal(x, y), f"unit {u} window {j} differs"
    run.assert_all_live()
    assert run.route_events >= 5
    other.close()


def test_restore_refuses_what_it_cannot_take():
    import torch
    wl = WL
    stream = torch.cuda.current_stream().cuda_stream
    a = qe.QECache(qe.config_from_workload(wl, batch=wl.batch, n_layers=1), stream)
    K, V = host_kv(wl, 0, 0, 64, wl.batch)
    a.qe_append(0, to_dev(K), to_dev(V), 64)
    snap = a.snapshot()
    # another configuration (a longer max_context: other table sizes)
    b = qe.QECache(qe.config_from_workload(wl, batch=wl.batch, n_layers=1,
                                           max_context=wl.prefill + wl.decode_steps + 512), stream)
    with pytest.raises(qe.QEError) as e:
        b.restore(snap)
    assert e.value.status == qe.QE_ERR_INVALID_ARG
    # a damaged header
    bad = snap.copy()
    bad[0] ^= 0xFF
    with pytest.raises(qe.QEError) as e:
        a.restore(bad)
    assert e.value.status == qe.QE_ERR_INVALID_ARG
    # a truncated snapshot
    with pytest.raises(qe.QEError) as e:
        a.restore(snap[: snap.nbytes // 2])
    assert e.value.status == qe.QE_ERR_INVALID_ARG
    # a layer awaiting qe_verify_commit
    n_q = 2
    Kd = np.stack([host_kv(wl, 0, 64 + j, 1, wl.batch)[0][:, :, 0] for j in range(n_q)])
    Vd = np.stack([host_kv(wl, 0, 64 + j, 1, wl.batch)[1][:, :, 0] for j in range(n_q)])
    Qd = np.stack([host_q(wl, 0, 1 + j, wl.batch) for j in range(n_q)])
    out = torch.empty(n_q, wl.batch, wl.n_q_heads, wl.head_dim, device="cuda", dtype=torch.float32)
    a.qe_verify(0, to_dev(Qd), to_dev(Kd), to_dev(Vd), out, n_q)
    with pytest.raises(qe.QEError) as e:
        a.snapshot()
    assert e.value.status == qe.QE_ERR_STATE
    a.qe_verify_commit(0, n_q)
    assert a.snapshot().nbytes == snap.nbytes       # the same layout
    # the restore still takes the earlier snapshot (length back to 64)
    a.restore(snap)
    assert a.layer_info(0).length == 64
    a.close()
    b.close()
    # a five-tier handle
    tw = gen.WORKLOADS["tiny_hqe"]
    c = qe.QECache(qe.config_from_workload(tw), stream)
    with pytest.raises(qe.QEError) as e:
        c.snapshot()
    assert e.value.status == qe.QE_ERR_STATE
    c.close()
