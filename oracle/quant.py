"""Uniform min/scale quantizer and KIVI's asymmetric quantization axes.

Test infrastructure (see ``oracle/__init__``).

Sources
-------
* HqeKV reading notes (zhongzhuzhou.org, 2026-08-26), §2.3 eq. (2): a group
  ``X`` is mapped with offset ``z = min(X)`` and scale
  ``s = (max(X) - min(X)) / (2^b - 1)``; ``X_q = (X - z) / s`` and
  ``X_dq = X_q * s + z``; each value goes to the nearest of the 2^b levels.
* QEvict reading notes (zhongzhuzhou.org, 2026-08-08), §1 "low-bit KV
  quantization" and Algorithm 1 (lines on first demotion): keys are
  quantized per channel, values per token (KIVI's asymmetric scheme), once
  per window, and the codes plus scale/zero are kept in a ledger.
* KV Cache technology evolution (zane-jiang.github.io), §5: KIVI groups
  keys along channels across tokens and values along each token.

Readings where the pages are silent:
* rounding is to nearest with ties to even (``np.rint``), codes clipped to
  ``[0, 2^b - 1]``;
* the scale and the normalised value are computed in float32 with IEEE
  division; a constant group (``s == 0``) gets all-zero codes;
* dequantization is ``code * s + z`` evaluated in float64 from the float32
  parameters;
* a window's key groups span only its valid tokens (window 0 excludes the
  sink tokens); a value group spans ``v_group`` channels of one token.
"""
from __future__ import annotations

import dataclasses

import numpy as np

F32 = np.float32


def uniform_quantize(x, bits: int, axis: int):
    """eq. (2) along ``axis``: returns (codes uint8, z float32, s float32).

    ``x`` is float32; ``z`` and ``s`` keep a size-1 ``axis``.
    """
    x = np.asarray(x, dtype=F32)
    levels = F32(2 ** bits - 1)
    z = np.min(x, axis=axis, keepdims=True)
    mx = np.max(x, axis=axis, keepdims=True)
    s = (mx - z) / levels                      # float32 subtract, float32 IEEE divide
    safe = np.where(s == 0, F32(1), s)
    xq = (x - z) / safe                        # float32
    codes = np.clip(np.rint(xq), F32(0), levels)
    codes = np.where(s == 0, F32(0), codes)
    return codes.astype(np.uint8), z.astype(F32), s.astype(F32)


def uniform_dequantize(codes, z, s):
    """X_dq = X_q * s + z, in float64."""
    return codes.astype(np.float64) * np.asarray(s, np.float64) + np.asarray(z, np.float64)


@dataclasses.dataclass
class QuantizedWindow:
    """Ledger entry of one window: INT2 codes and float32 parameters.

    k_codes [n, d] (per-channel groups over the window's n valid tokens),
    k_min/k_scale [d]; v_codes [n, d] (per-token groups of ``v_group``
    channels), v_min/v_scale [n, d // v_group].
    """
    k_codes: np.ndarray
    k_min: np.ndarray
    k_scale: np.ndarray
    v_codes: np.ndarray
    v_min: np.ndarray
    v_scale: np.ndarray
    v_group: int

    def dequantize(self):
        """Reconstructed (K, V) as float64 [n, d]."""
        k = uniform_dequantize(self.k_codes, self.k_min[None, :], self.k_scale[None, :])
        n, d = self.v_codes.shape
        g = self.v_group
        vc = self.v_codes.reshape(n, d // g, g)
        v = uniform_dequantize(vc, self.v_min[:, :, None], self.v_scale[:, :, None]).reshape(n, d)
        return k, v

    def equal(self, other: "QuantizedWindow") -> bool:
        return all(np.array_equal(getattr(self, f), getattr(other, f)) for f in
                   ("k_codes", "k_min", "k_scale", "v_codes", "v_min", "v_scale"))


def kivi_quantize_window(k, v, bits: int = 2, v_group: int | None = None) -> QuantizedWindow:
    """Quantize one window's valid tokens: keys per channel, values per token.

    ``k`` and ``v`` are the original bf16 values as float32 arrays [n, d].
    """
    k = np.asarray(k, dtype=F32)
    v = np.asarray(v, dtype=F32)
    n, d = k.shape
    g = d if v_group is None else v_group
    assert d % g == 0
    kc, kz, ks = uniform_quantize(k, bits, axis=0)            # one group per channel
    vv = v.reshape(n, d // g, g)
    vc, vz, vs = uniform_quantize(vv, bits, axis=2)           # one group per token (and channel group)
    return QuantizedWindow(kc, kz[0], ks[0], vc.reshape(n, d), vz[:, :, 0], vs[:, :, 0], g)
