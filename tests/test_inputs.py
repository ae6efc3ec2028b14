"""The seeded input generator (no GPU): published SplitMix64 outputs, distribution, bf16 rounding."""
import numpy as np
import pytest
import torch

import qe_inputs as gen


def test_splitmix64_reference_sequence():
    # SplitMix64 generator seeded with 1234567: outputs are mix(seed + k * gamma), k = 1, 2, ...
    seed = 1234567
    got = [int(gen.splitmix64(np.uint64((seed + (k - 1) * gen.GAMMA) % 2 ** 64))) for k in range(1, 6)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_normals_moments_and_support():
    keys = gen.row_key(99, gen.T_K, 0, 0, 0, np.arange(4096))
    z = gen.normal_rows_f32(keys, 128).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1) < 0.01
    assert np.abs(z).max() <= 6
    # excess kurtosis of an Irwin-Hall(12) sum is -0.1
    k = ((z - z.mean()) ** 4).mean() / z.var() ** 2 - 3
    assert -0.2 < k < 0.0


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(100000).astype(np.float32) * 10
    # exact ties: values with the low 16 bits = 0x8000
    ties = (rng.integers(0, 2 ** 31, 1000, dtype=np.int64).astype(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    ties = ties.view(np.float32)
    ties = ties[np.isfinite(ties)]
    for arr in (x, ties):
        mine = gen.bf16_bits_rne(arr)
        ref = torch.from_numpy(arr).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(mine, ref)


def test_workload_geometry():
    for wl in gen.WORKLOADS.values():
        assert wl.n_q_heads % wl.n_kv_heads == 0
        assert wl.head_dim in (64, 128) and wl.window % 16 == 0
        assert 0 <= wl.n_sink < wl.window
    wl = gen.WORKLOADS["throughput_32k"]
    ch = gen.outlier_channels(wl, 3, 5)
    assert len({c for c, _ in ch}) == 4 and all(m == 10 for _, m in ch)
    kb, vb = gen.gen_keys_values(wl, 2, 3, 5, 1000, 64)
    k = gen.bf16_bits_to_f32(kb)
    big = [c for c, _ in ch]
    small = [c for c in range(128) if c not in big]
    assert k[:, big].std() > 5 * k[:, small].std()


def test_queries_and_drift_are_deterministic():
    wl = gen.WORKLOADS["llama8b_stack"]
    a = gen.gen_queries(wl, 0, 7, range(8, 12), 5)
    b = gen.gen_queries(wl, 0, 7, range(8, 12), 5)
    assert np.array_equal(a, b)
    j = gen.drift_window(wl, 0, 7, 2, 5)
    assert 0 <= j < wl.prefill // wl.window
    assert gen.drift_window(wl, 0, 7, 2, 64) == j          # same epoch (steps 1..64)
    mu = gen.drift_mean(wl, 0, 7, 2, 5)
    kb, _ = gen.gen_keys_values(wl, 0, 7, 2, j * wl.window, wl.window)
    assert np.allclose(mu, gen.bf16_bits_to_f32(kb).astype(np.float64).mean(0), rtol=0, atol=1e-12)
