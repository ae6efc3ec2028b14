"""Pins of the RoPE step (keys stored pre-RoPE, rotated at original positions) against closed
forms and the mathematics of rotations."""
import math

import numpy as np

import qe_inputs as gen
from oracle.rope import apply_rope, rope_angles
from oracle.run import make_unit


def test_direction_pairing_and_frequencies():
    # d = 2: theta_0 = 1, (1, 0) rotates to (cos p, sin p)
    for p in (0, 1, 7, 1000):
        assert np.allclose(apply_rope([[1.0, 0.0]], [p], 10000.0), [[math.cos(p), math.sin(p)]], atol=1e-12)
    # d = 4: channels (2, 3) are pair 1 with theta_1 = base^(-1/2) = 1/100
    r = apply_rope([[0.0, 0.0, 1.0, 0.0]], [300], 10000.0)
    assert np.allclose(r, [[0.0, 0.0, math.cos(3.0), math.sin(3.0)]], atol=1e-12)
    assert np.allclose(rope_angles([5], 8, 10000.0), [[5.0, 0.5, 0.05, 0.005]])
    x = np.random.default_rng(0).standard_normal((3, 16))
    assert np.array_equal(apply_rope(x, [0, 0, 0], 10000.0), x)


def test_relative_position_and_norms():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 64))
    k = rng.standard_normal((1, 64))
    for t, p in ((100, 3), (5, 5), (70000, 12345)):
        a = apply_rope(q, [t], 10000.0) @ apply_rope(k, [p], 10000.0).T
        b = apply_rope(q, [t + 977], 10000.0) @ apply_rope(k, [p + 977], 10000.0).T
        assert abs(a - b) < 1e-9 * (1 + abs(a))
        c = q @ apply_rope(k, [p - t], 10000.0).T
        assert abs(a - c) < 1e-9 * (1 + abs(a))
    r = apply_rope(k, [123], 10000.0)
    assert np.allclose(np.hypot(r[0, 0::2], r[0, 1::2]), np.hypot(k[0, 0::2], k[0, 1::2]), rtol=1e-13)


def test_uncompressed_unit_attends_over_rotated_keys():
    # a unit that keeps every window Full attends exactly as softmax(q . R_p k / sqrt(d)), with
    # the rotation written as multiplication of complex numbers x + iy by exp(i p theta)
    import dataclasses
    wl = dataclasses.replace(gen.WORKLOADS["tiny_qevict"], kf=100, kq=0, rope_theta=10000.0, plant_tokens=())
    u = make_unit(wl)
    kb, vb = gen.gen_keys_values(wl, 0, 0, 0, 0, 100)
    K, V = gen.bf16_bits_to_f32(kb).astype(np.float64), gen.bf16_bits_to_f32(vb).astype(np.float64)
    u.append(K[:99], V[:99])
    q = gen.bf16_bits_to_f32(gen.gen_queries(wl, 0, 0, range(4), 1)).astype(np.float64)
    o, _, _ = u.decode_step(q, K[99:], V[99:])
    d = K.shape[1]
    theta = 10000.0 ** (-np.arange(d // 2) * 2.0 / d)
    z = (K[:, 0::2] + 1j * K[:, 1::2]) * np.exp(1j * np.arange(100)[:, None] * theta[None, :])
    Kr = np.empty_like(K)
    Kr[:, 0::2], Kr[:, 1::2] = z.real, z.imag
    lg = q @ Kr.T / math.sqrt(d)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    assert np.allclose(o, p @ V, rtol=1e-10, atol=1e-12)
