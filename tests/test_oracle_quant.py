"""Pins of the eq. (2) quantizer and the KIVI axes (no GPU).

eq. (2) (HqeKV reading notes, §2.3) states z = min, s = (max - min)/(2^b - 1)
and that every value goes to the nearest level; the tests check the codes
against that nearest-level statement computed independently in float64, plus
the closed forms (min reproduced exactly, grid values round-trip, error at
most s/2).
"""
import numpy as np
import pytest

from oracle.quant import kivi_quantize_window, uniform_dequantize, uniform_quantize

RNG = np.random.default_rng(7)


def _groups():
    yield RNG.standard_normal((64, 32)).astype(np.float32)
    yield (RNG.standard_normal((16, 128)) * np.array([8.0] * 3 + [1.0] * 125)).astype(np.float32)
    yield RNG.uniform(-1e-3, 1e-3, (8, 17)).astype(np.float32)
    yield np.round(RNG.standard_normal((32, 64)) * 4).astype(np.float32) / 4   # many ties


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_codes_are_nearest_levels(bits):
    for x in _groups():
        codes, z, s = uniform_quantize(x, bits, axis=1)
        lv = np.arange(2 ** bits, dtype=np.float64)
        levels = z.astype(np.float64) + lv[None, :] * s.astype(np.float64)          # [g, L]
        dist = np.abs(x.astype(np.float64)[:, :, None] - levels[:, None, :])         # [g, n, L]
        best = dist.min(axis=2)
        chosen = np.take_along_axis(dist, codes[:, :, None].astype(np.int64), 2)[:, :, 0]
        # float32 evaluation of (x - z)/s may flip an exact midpoint: allow that slack only
        slack = 4 * np.finfo(np.float32).eps * (np.abs(x) + np.abs(z) + s).astype(np.float64)
        assert np.all(chosen <= best + slack)


def test_min_reproduced_and_error_bound():
    for x in _groups():
        codes, z, s = uniform_quantize(x, 2, axis=1)
        xh = uniform_dequantize(codes, z, s)
        amin = np.argmin(x, axis=1)
        rows = np.arange(x.shape[0])
        assert np.all(codes[rows, amin] == 0)
        assert np.array_equal(xh[rows, amin], x[rows, amin].astype(np.float64))
        amax = np.argmax(x, axis=1)
        assert np.all(codes[rows, amax] == 3)
        bound = s.astype(np.float64) / 2 + 4 * np.finfo(np.float32).eps * (np.abs(x) + s)
        assert np.all(np.abs(xh - x) <= bound)
        assert np.all((codes >= 0) & (codes <= 3))


def test_constant_group_and_grid_roundtrip():
    x = np.full((3, 9), 1.625, np.float32)
    codes, z, s = uniform_quantize(x, 2, axis=1)
    assert np.all(codes == 0) and np.all(s == 0) and np.all(z == 1.625)
    assert np.array_equal(uniform_dequantize(codes, z, s), x.astype(np.float64))
    # values exactly on a power-of-two grid come back exactly
    c = RNG.integers(0, 4, (5, 40))
    c[:, 0], c[:, 1] = 0, 3
    zz, ss = -0.75, 0.125
    x = (zz + c * ss).astype(np.float32)
    codes, z, s = uniform_quantize(x, 2, axis=1)
    assert np.array_equal(codes, c.astype(np.uint8))
    assert np.array_equal(uniform_dequantize(codes, z, s), x.astype(np.float64))


def test_half_steps_round_to_even():
    # z = 0, s = 1: (x - z)/s = 0.5, 1.5, 2.5 are exact midpoints
    x = np.array([[0.0, 3.0, 0.5, 1.5, 2.5]], np.float32)
    codes, z, s = uniform_quantize(x, 2, axis=1)
    assert s[0, 0] == 1.0
    assert codes.tolist() == [[0, 3, 0, 2, 2]]


def test_kivi_axes():
    n, d = 32, 64
    k = RNG.standard_normal((n, d)).astype(np.float32)
    v = RNG.standard_normal((n, d)).astype(np.float32)
    q = kivi_quantize_window(k, v)
    assert q.k_codes.shape == (n, d) and q.k_min.shape == (d,) and q.v_min.shape == (n, 1)
    # keys: one group per channel over the window's tokens
    assert np.array_equal(q.k_min, k.min(axis=0))
    # values: one group per token over its channels
    assert np.array_equal(q.v_min[:, 0], v.min(axis=1))
    # changing one channel of the keys leaves the other channels' codes alone
    k2 = k.copy()
    k2[:, 5] = k2[:, 5] ** 3 + 2
    q2 = kivi_quantize_window(k2, v)
    others = [c for c in range(d) if c != 5]
    assert np.array_equal(q.k_codes[:, others], q2.k_codes[:, others])
    assert np.array_equal(q.k_min[others], q2.k_min[others]) and q.k_min[5] != q2.k_min[5]
    # a positive rescale of a group leaves its codes unchanged (codes depend on (x - min)/range only)
    k3 = k.copy()
    k3[:, 9] *= 4
    assert np.array_equal(kivi_quantize_window(k3, v).k_codes, q.k_codes)
    # changing one token of the values leaves the other tokens' codes alone
    v2 = v.copy()
    v2[3] = v2[3] * 5 + 1
    q3 = kivi_quantize_window(k, v2)
    rows = [i for i in range(n) if i != 3]
    assert np.array_equal(q.v_codes[rows], q3.v_codes[rows])
    # dequantized values stay within half a step of the originals on both axes
    kh, vh = q.dequantize()
    assert np.all(np.abs(kh - k) <= q.k_scale[None, :] / 2 + 1e-6)
    assert np.all(np.abs(vh - v) <= q.v_scale / 2 + 1e-6)


def test_kivi_value_groups():
    n, d = 8, 128
    k = RNG.standard_normal((n, d)).astype(np.float32)
    v = RNG.standard_normal((n, d)).astype(np.float32)
    q = kivi_quantize_window(k, v, v_group=32)
    assert q.v_min.shape == (n, 4)
    assert np.array_equal(q.v_min, v.reshape(n, 4, 32).min(axis=2))
