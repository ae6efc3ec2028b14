"""Rotary position embedding applied to stored pre-RoPE keys at their original positions.

Test infrastructure (see ``oracle/__init__``).

Sources
-------
* QEvict reading notes, §4.4 (Algorithm 1, promotion): keys are quantized in the pre-RoPE
  domain and stored with their original absolute positions; the rotation is applied again with
  those positions, so the position information never passes through the lossy codes.
* KV Cache technology evolution, §5 (KVQuant) and §10.3: pre-rotation keys must keep their
  original position semantics; re-applying RoPE with compacted slot numbers would change the
  relative distances the model sees.

Readings where the pages are silent:
* RoPE is the original rotary embedding: channel pairs (2i, 2i + 1), i = 0 .. d/2 - 1, are
  rotated by the angle p * theta_i, theta_i = base^(-2i / d), base 10000 unless configured,
  (x, y) -> (x cos - y sin, x sin + y cos);
* queries reach the cache already rotated at their own position (the model's usual query);
  keys are appended and stored pre-RoPE, and every key -- bf16 or dequantized -- is rotated at
  its original position when it is attended to; all in float64.
"""
from __future__ import annotations

import numpy as np


def rope_angles(positions, d: int, base: float) -> np.ndarray:
    """[n, d/2] angles p * theta_i (float64)."""
    p = np.asarray(positions, np.float64).reshape(-1, 1)
    i = np.arange(d // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / d)
    return p * theta[None, :]


def apply_rope(x, positions, base: float) -> np.ndarray:
    """Rotate rows of x [n, d] (float64 result) by their positions."""
    x = np.asarray(x, np.float64)
    n, d = x.shape
    a = rope_angles(positions, d, base)
    c, s = np.cos(a), np.sin(a)
    out = np.empty_like(x)
    out[:, 0::2] = x[:, 0::2] * c - x[:, 1::2] * s
    out[:, 1::2] = x[:, 0::2] * s + x[:, 1::2] * c
    return out
