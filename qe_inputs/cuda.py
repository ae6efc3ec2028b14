"""GPU twin of the qe_inputs generator (``_gen.so``, built from ``gen.cu``).

Produces exactly the bits of :func:`qe_inputs.gen_keys_values` and
:func:`qe_inputs.gen_queries` (workloads without a planted direction) directly in device
memory, for workloads too large to generate on the host.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import T_K, T_V, Workload, channel_scales

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_gen.so")
_lib = None


def build() -> str:
    import sys
    sys.path.insert(0, os.path.dirname(_HERE))
    from tiered_quantize_evict_gb300.build import compile_units
    return compile_units([os.path.join(_HERE, "gen.cu")], LIB_PATH, [_HERE])


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} missing: build it with qe_inputs.cuda.build()")
        L = ctypes.CDLL(LIB_PATH)
        I, P, U = ctypes.c_int, ctypes.c_void_p, ctypes.c_ulonglong
        L.qe_gen_rows.argtypes = [U, I, I, I, I, I, I, I, P, P, P]
        L.qe_gen_rows.restype = I
        L.qe_gen_queries.argtypes = [U, I, I, I, I, I, I, I, I, I, P, P, P]
        L.qe_gen_queries.restype = I
        _lib = L
    return _lib


class DeviceGenerator:
    """Keeps per-layer key channel scales on the device and fills bf16 (int16-typed) tensors."""

    def __init__(self, wl: Workload, device="cuda"):
        import torch
        if wl.plant_tokens:
            raise ValueError("planted-direction workloads are generated on the host")
        self.wl = wl
        self.torch = torch
        self.scales = {}
        self.device = device

    def _kscale(self, layer: int):
        if layer not in self.scales:
            s = np.stack([channel_scales(self.wl, layer, h) for h in range(self.wl.n_kv_heads)]).astype(np.int32)
            self.scales[layer] = self.torch.from_numpy(s).to(self.device)
        return self.scales[layer]

    def keys_values(self, layer: int, pos0: int, n: int, k_out, v_out, stream: int = 0):
        """k_out, v_out: [B][H_kv][n][d] int16/bfloat16 device tensors."""
        wl = self.wl
        L = lib()
        rc = L.qe_gen_rows(wl.seed, T_K, wl.batch, layer, wl.n_kv_heads, pos0, n, wl.head_dim,
                           self._kscale(layer).data_ptr(), k_out.data_ptr(), stream)
        rc |= L.qe_gen_rows(wl.seed, T_V, wl.batch, layer, wl.n_kv_heads, pos0, n, wl.head_dim,
                            None, v_out.data_ptr(), stream)
        if rc:
            raise RuntimeError(f"generator launch failed ({rc})")

    def queries(self, layer: int, step: int, q_out, stream: int = 0):
        """q_out: [B][H_q][d] device tensor for decode step ``step`` (1-based)."""
        wl = self.wl
        rc = lib().qe_gen_queries(wl.seed, wl.batch, layer, wl.n_q_heads, wl.group, step, wl.head_dim,
                                  wl.drift_period, wl.prefill, wl.window, self._kscale(layer).data_ptr(),
                                  q_out.data_ptr(), stream)
        if rc:
            raise RuntimeError(f"generator launch failed ({rc})")
