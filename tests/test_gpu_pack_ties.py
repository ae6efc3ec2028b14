"""The 2-bit packer on rounding ties and scale extremes (GPU).

eq. (2) rounds (x - z) / s to the nearest level, ties to even.  The packer estimates the quotient
and takes the correctly rounded division only near a half-integer or for a scale outside
[1e-30, 1e30].  This test plants, in every key channel and value row of the windows that get
packed, bf16 values whose float32 quotient is exactly a half-integer, plus groups with tiny and
huge scales and constant groups (s = 0), and compares the codes and the float32 parameters bit
for bit with the oracle's quantizer.
"""
import numpy as np
import pytest

from oracle.quant import kivi_quantize_window

pytestmark = pytest.mark.gpu

W, D, NWIN, SINK = 32, 128, 12, 5


def _bf16(x):
    """x rounded to the nearest bf16 value (ties to even), as float32."""
    b = int(np.float32(x).view(np.uint32))
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return np.uint32(b).view(np.float32)


# (min, max) of a group; bf16-exact.  Exact scales, inexact scales, a scale below 1e-30 and one
# above 1e30 (both take the correctly rounded division).
RANGES = [(_bf16(a), _bf16(b)) for a, b in [(0.0, 3.0), (-1.25, 4.75), (-5.0, 7.0), (-2.2, 5.9), (0.0, 0.7),
                                            (-1e-3, 2e-3), (0.0, 3 * 2.0 ** -110), (0.0, 3 * 2.0 ** 100)]]
BITS = np.arange(0, 1 << 16, dtype=np.uint32)
GRID = np.unique((BITS << 16).view(np.float32)[np.isfinite((BITS << 16).view(np.float32))])


def _group(lo, hi, rng, n):
    """n values: lo, hi, every bf16 value in [lo, hi] whose float32 quotient (x - lo) / s sits
    exactly on a half-integer, then random bf16 values of the range."""
    g = GRID[(GRID >= lo) & (GRID <= hi)]
    s = np.float32((hi - lo) / np.float32(3))
    q = (g - lo) / s
    ties = g[q - np.floor(q) == np.float32(0.5)]
    assert ties.size > 0, (lo, hi)
    pick = np.concatenate([[lo, hi], ties, g[rng.integers(0, g.size, n)]])[:n]
    return rng.permutation(pick).astype(np.float32)


def _bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_packer_ties_and_scale_extremes_match_ieee_division():
    import torch
    import tiered_quantize_evict_gb300 as qe
    rng = np.random.default_rng(7)
    L = W * NWIN
    K = np.full((L, D), 0.25, np.float32)
    V = np.full((L, D), 0.25, np.float32)
    for j in range(NWIN):
        rows = np.arange(j * W + (SINK if j == 0 else 0), (j + 1) * W)
        for c in range(D):                            # key groups: one channel over the window's tokens
            lo, hi = RANGES[(j + c) % len(RANGES)]
            K[rows, c] = _group(lo, hi, rng, rows.size)
        for r in rows:                                # value groups: one token over its channels
            lo, hi = RANGES[(j + r) % len(RANGES)]
            V[r] = _group(lo, hi, rng, D)
        K[rows, j] = 1.5                              # a constant key channel (s = 0) ...
        V[rows[j % rows.size]] = -0.75                # ... and a constant value row
    cfg = qe.QEConfig(batch=1, n_layers=1, n_q_heads=4, n_kv_heads=1, head_dim=D, window=W, route_period=1,
                      n_sink=SINK, n_recent=32, max_context=L + 8, cap_mode=0, kf=2, kq=8, frac_bf16=0.0,
                      frac_int2=0.0, budget_frac=0.0, out_fp32=1)
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    cache = qe.QECache(cfg, stream.cuda_stream)
    kt = torch.from_numpy(_bits(K).view(np.int16)).reshape(1, 1, L, D).to(dev)
    vt = torch.from_numpy(_bits(V).view(np.int16)).reshape(1, 1, L, D).to(dev)
    cache.qe_append(0, kt, vt, L)
    info = cache.layer_info(0)
    S = np.zeros((info.units, info.max_windows), np.float32)
    S[0, :NWIN] = np.arange(NWIN, 0, -1, dtype=np.float32)   # windows 0, 1 Full; 2..9 2-bit; 10 evicted
    cache.set_scores(0, S)
    cache.qe_route(0)
    tiers = cache.tiers(0)[0]
    quant = [j for j in range(NWIN) if tiers[j] == qe.TIER_QUANT]
    assert quant == list(range(2, 10)), tiers[:NWIN]
    for j in quant:
        ref = kivi_quantize_window(K[j * W:(j + 1) * W], V[j * W:(j + 1) * W])
        kc, vc, kz, ks, vz, vs = cache.quant_window(0, 0, j)
        assert np.array_equal(kz.view(np.uint32), ref.k_min.view(np.uint32)), f"window {j}: key min"
        assert np.array_equal(ks.view(np.uint32), ref.k_scale.view(np.uint32)), f"window {j}: key scale"
        assert np.array_equal(vz.view(np.uint32), ref.v_min[:, 0].view(np.uint32)), f"window {j}: value min"
        assert np.array_equal(vs.view(np.uint32), ref.v_scale[:, 0].view(np.uint32)), f"window {j}: value scale"
        bad = np.argwhere(kc != ref.k_codes)
        assert bad.size == 0, f"window {j}: key codes differ at {bad[:4].tolist()}"
        bad = np.argwhere(vc != ref.v_codes)
        assert bad.size == 0, f"window {j}: value codes differ at {bad[:4].tolist()}"
        assert (ks == 0).any() and (vs == 0).any() and (ks < 1e-30).any() and (ks > 1e30).any()
    cache.qe_synchronize()
