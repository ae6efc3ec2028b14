"""Speculative verify with rollback on the GPU against the oracle (H2O page §5, speculative
decoding): decode steps, verifies of several drafts with seeded acceptance counts (all, some,
none), and routing events interleave; every draft query's output, the scores after each commit,
the tiers after each routing event, and the 2-bit codes and bf16 windows are compared.

Keys used as stored may take the fused path (all drafts against one read of the cache on the
tensor cores, up to 64 draft x head rows); keys stored pre-RoPE verify draft by draft.  Every case
runs with the automatic choice and, where keys are used as stored, with each path forced, with up
to 16 drafts (64 rows at G = 4), head dims 64 and 128, windows 16, 32 and 64."""
import dataclasses

import numpy as np
import pytest

import qe_inputs as gen
import tiered_quantize_evict_gb300 as qe
from qe_testlib import OUT_TOL, TIER_CODE, ParityRun, host_kv, host_q, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    "d128_w32_g4": dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="verify_d128", batch=2, n_q_heads=8,
                                       n_kv_heads=2, head_dim=128, prefill=290, decode_steps=60, window=32,
                                       route_period=12, n_sink=5, n_recent=32, kf=4, kq=6, plant_tokens=(),
                                       seed=51),
    "d64_w16_g2_rope": dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="verify_d64", batch=1, n_q_heads=4,
                                           n_kv_heads=2, head_dim=64, prefill=150, decode_steps=60, window=16,
                                           route_period=8, n_sink=3, n_recent=16, kf=3, kq=4, plant_tokens=(),
                                           rope_theta=10000.0, seed=52),
    # fused path at its limits: 16 drafts x 4 heads = 64 rows
    "d128_w32_g4_16drafts": dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="verify_d128_16",
                                                batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, prefill=420,
                                                decode_steps=320, window=32, route_period=12, n_sink=5, n_recent=32,
                                                kf=4, kq=6, plant_tokens=(), seed=53),
    "d64_w16_g2_16drafts": dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="verify_d64_16", batch=1,
                                               n_q_heads=4, n_kv_heads=2, head_dim=64, prefill=150, decode_steps=320,
                                               window=16, route_period=8, n_sink=3, n_recent=16, kf=3, kq=4,
                                               plant_tokens=(), seed=54),
    "d128_w64_g1_16drafts": dataclasses.replace(gen.WORKLOADS["tiny_qevict"], name="verify_d128_w64", batch=3,
                                                n_q_heads=1, n_kv_heads=1, head_dim=128, prefill=700,
                                                decode_steps=320, window=64, route_period=16, n_sink=0, n_recent=20,
                                                kf=2, kq=4, plant_tokens=(), seed=55),
}
MAX_DRAFTS = {"d128_w32_g4_16drafts": 16, "d64_w16_g2_16drafts": 16, "d128_w64_g1_16drafts": 16}


PATHS = {"auto": 0, "fused": 1, "per_draft": 2}


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("name", sorted(CASES))
def test_verify_commit_trajectory(name, path):
    import torch
    wl = CASES[name]
    if wl.rope_theta and path != "auto":
        pytest.skip("keys stored pre-RoPE always verify draft by draft")
    track = [(b, 0, h) for b in range(wl.batch) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, 1, track)
    assert qe.debug_inject(qe.QE_DEBUG_VERIFY_PATH, PATHS[path], run.cache) == 0
    run.prefill()
    rng = np.random.default_rng(7)
    cache, G, D = run.cache, wl.group, wl.head_dim
    n_verifies = 0
    last_route = 0
    for event in range(14):
        if event % 3 == 2:
            run.step(check=True)                          # an ordinary decode step between verifies
        else:
            n_q = int(rng.integers(1, MAX_DRAFTS.get(name, 4) + 1))
            acc = int(rng.integers(0, n_q + 1))
            t0, L0 = run.t, wl.prefill + run.t
            K = np.stack([host_kv(wl, 0, L0 + j, 1, wl.batch)[0][:, :, 0] for j in range(n_q)])
            V = np.stack([host_kv(wl, 0, L0 + j, 1, wl.batch)[1][:, :, 0] for j in range(n_q)])
            Q = np.stack([host_q(wl, 0, t0 + 1 + j, wl.batch) for j in range(n_q)])
            out = torch.empty(n_q, wl.batch, wl.n_q_heads, D, device=run.dev, dtype=torch.float32)
            cache.qe_verify(0, to_dev(Q), to_dev(K), to_dev(V), out, n_q)
            got = out.cpu().numpy().astype(np.float64)
            for tr in run.tracked:
                qs = [gen.bf16_bits_to_f32(Q[j, tr.b, tr.kvh * G:(tr.kvh + 1) * G]) for j in range(n_q)]
                ks = [gen.bf16_bits_to_f32(K[j, tr.b, tr.kvh]) for j in range(n_q)]
                vs = [gen.bf16_bits_to_f32(V[j, tr.b, tr.kvh]) for j in range(n_q)]
                outs, _ = tr.unit.verify(qs, ks, vs)
                for j in range(n_q):
                    for i in range(G):
                        ref = outs[j][i]
                        err = np.linalg.norm(got[j, tr.b, tr.kvh * G + i] - ref) / np.linalg.norm(ref)
                        run.max_out_err = max(run.max_out_err, err)
                        assert err <= OUT_TOL, f"verify {event} draft {j} unit {(tr.b, tr.kvh)}: rel-L2 {err:.2e}"
            cache.qe_verify_commit(0, acc)
            for tr in run.tracked:
                tr.unit.commit(acc)
            run.t += acc
            n_verifies += 1
            run.check_scores()
            info = cache.layer_info(0)
            assert info.length == wl.prefill + run.t
            tiers = cache.tiers(0)
            for tr in run.tracked:
                u = tr.b * wl.n_kv_heads + tr.kvh
                for j in range(info.max_windows):
                    want = TIER_CODE[tr.unit.tier[j]] if j in tr.unit.tier else 0
                    assert tiers[u, j] == want, f"verify {event} unit {u} window {j}: {tiers[u, j]} vs {want}"
        if run.t // wl.route_period > last_route:           # a routing event once per period
            last_route = run.t // wl.route_period
            run.route_and_check()
            for tr in run.tracked:
                if tr.live:
                    run.check_bf16_windows(tr)
    cache.qe_synchronize()
    assert n_verifies >= 8 and run.route_events >= 2
    print(f"{name}: verifies {n_verifies}, routes {run.route_events}, max out rel-L2 {run.max_out_err:.2e}, "
          f"max score rel {run.max_score_err:.2e}, codes {run.codes_checked}")


def test_rejected_draft_returns_its_window_slot():
    """Drafts cross a window boundary and only the first is kept: the window the second opened
    closes (its slot goes back to the free list) and the next decode step opens it again."""
    import torch
    wl = dataclasses.replace(CASES["d128_w32_g4"], name="verify_boundary", prefill=287)
    track = [(b, 0, h) for b in range(wl.batch) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, 1, track)
    run.prefill()
    cache = run.cache
    n_q, L0 = 3, wl.prefill
    K = np.stack([host_kv(wl, 0, L0 + j, 1, wl.batch)[0][:, :, 0] for j in range(n_q)])
    V = np.stack([host_kv(wl, 0, L0 + j, 1, wl.batch)[1][:, :, 0] for j in range(n_q)])
    Q = np.stack([host_q(wl, 0, 1 + j, wl.batch) for j in range(n_q)])
    out = torch.empty(n_q, wl.batch, wl.n_q_heads, wl.head_dim, device=run.dev, dtype=torch.float32)
    cache.qe_verify(0, to_dev(Q), to_dev(K), to_dev(V), out, n_q)
    assert (cache.tiers(0)[:, 9] == 1).all()           # window 9 opened (Pinned) by draft 1
    cache.qe_verify_commit(0, 1)
    for tr in run.tracked:
        tr.unit.verify([gen.bf16_bits_to_f32(Q[j, tr.b, tr.kvh * wl.group:(tr.kvh + 1) * wl.group])
                        for j in range(n_q)],
                       [gen.bf16_bits_to_f32(K[j, tr.b, tr.kvh]) for j in range(n_q)],
                       [gen.bf16_bits_to_f32(V[j, tr.b, tr.kvh]) for j in range(n_q)])
        tr.unit.commit(1)
    run.t = 1
    assert (cache.tiers(0)[:, 9] == 0).all() and cache.layer_info(0).length == 288
    run.check_scores()
    for _ in range(3):                                   # window 9 opens again from the free list
        run.step()
    assert (cache.tiers(0)[:, 9] == 1).all()
    for tr in run.tracked:
        run.check_bf16_windows(tr)
    cache.qe_synchronize()


@pytest.mark.parametrize("host", ["pinned", "pageable"])
def test_fused_verify_host_buffers_bf16_outputs(host):
    """The fused path with every buffer in host memory (staged through the handle's buffers)
    and bf16 outputs: each draft's output against the oracle within 4e-3 relative L2 (bf16
    rounding of the outputs included), then the scores after each commit and the tiers after
    each routing event, as with device buffers."""
    wl = CASES["d128_w32_g4"]
    track = [(b, 0, h) for b in range(wl.batch) for h in range(wl.n_kv_heads)]
    run = ParityRun(wl, wl.batch, 1, track, host=host, out_fp32=False)
    assert qe.debug_inject(qe.QE_DEBUG_VERIFY_PATH, 1, run.cache) == 0
    run.prefill()
    cache, G, D = run.cache, wl.group, wl.head_dim
    rng = np.random.default_rng(11)
    last_route = 0
    for event in range(6):
        n_q = int(rng.integers(5, 17))
        acc = int(rng.integers(0, n_q + 1))
        t0, L0 = run.t, wl.prefill + run.t
        K = np.stack([host_kv(wl, 0, L0 + j, 1, wl.batch)[0][:, :, 0] for j in range(n_q)])
        V = np.stack([host_kv(wl, 0, L0 + j, 1, wl.batch)[1][:, :, 0] for j in range(n_q)])
        Q = np.stack([host_q(wl, 0, t0 + 1 + j, wl.batch) for j in range(n_q)])
        out = run.out_buffer((n_q, wl.batch, wl.n_q_heads, D))
        k_, v_, q_ = run._place(K), run._place(V), run._place(Q)
        cache.qe_verify(0, q_, k_, v_, out, n_q)
        cache.qe_synchronize()
        del k_, v_, q_
        got = run.read_buffer(out).astype(np.float64)
        for tr in run.tracked:
            qs = [gen.bf16_bits_to_f32(Q[j, tr.b, tr.kvh * G:(tr.kvh + 1) * G]) for j in range(n_q)]
            ks = [gen.bf16_bits_to_f32(K[j, tr.b, tr.kvh]) for j in range(n_q)]
            vs = [gen.bf16_bits_to_f32(V[j, tr.b, tr.kvh]) for j in range(n_q)]
            outs, _ = tr.unit.verify(qs, ks, vs)
            for j in range(n_q):
                for i in range(G):
                    ref = outs[j][i]
                    err = np.linalg.norm(got[j, tr.b, tr.kvh * G + i] - ref) / np.linalg.norm(ref)
                    run.max_out_err = max(run.max_out_err, err)
                    assert err <= 4e-3, f"verify {event} draft {j} unit {(tr.b, tr.kvh)}: rel-L2 {err:.2e}"
        cache.qe_verify_commit(0, acc)
        for tr in run.tracked:
            tr.unit.commit(acc)
        run.t += acc
        run.check_scores()
        assert cache.layer_info(0).length == wl.prefill + run.t
        if run.t // wl.route_period > last_route:
            last_route = run.t // wl.route_period
            run.route_and_check()
    cache.qe_synchronize()
    run.assert_all_live()
    print(f"{host}: max out rel-L2 {run.max_out_err:.2e}, max score rel {run.max_score_err:.2e}, "
          f"routes {run.route_events}")
