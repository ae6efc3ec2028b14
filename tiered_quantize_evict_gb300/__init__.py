"""Tiered (bf16 / 2-bit / evicted) KV-cache decode attention for GB300 (sm_103a).

Thin ctypes binding of the C ABI in ``include/qe.h`` (``_lib/libqe.so``).  Every step of
the decode path (append, attention with fused window scoring, routing, packing, moves)
runs in the library's CUDA kernels; this module only marshals pointers, sizes and status
codes.  Importing it does not load the library; the first call does, and raises if the
library has not been built (``python -m tiered_quantize_evict_gb300.build``) - there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libqe.so")

QE_OK, QE_ERR_INVALID_ARG, QE_ERR_OOM, QE_ERR_CAPACITY, QE_ERR_CUDA = 0, 1, 2, 3, 4
QE_ERR_TIMEOUT, QE_ERR_STATE, QE_ERR_HOST_STORE, QE_ERR_DEVICE = 5, 6, 7, 8
TIER_NONE, TIER_PINNED, TIER_FULL, TIER_QUANT, TIER_EVICTED = 0, 1, 2, 3, 4
QE_DEVICE_PTRS, QE_HOST_PTRS = 0, 1

EXPORTED = [
    "qe_init", "qe_destroy", "qe_last_error", "qe_append", "qe_decode_step", "qe_route",
    "qe_synchronize", "qe_get_layer_info", "qe_get_tiers", "qe_get_scores", "qe_set_scores",
    "qe_get_quant_window", "qe_get_bf16_window", "qe_get_route_stats", "qe_set_timing",
    "qe_get_timing", "qe_kernel_launches", "qe_decode_step_noalloc", "qe_get_route_diag",
    "qe_get_token_tiers", "qe_get_token_scores", "qe_get_token_counts", "qe_get_token",
    "qe_verify", "qe_verify_commit", "qe_debug_inject", "qe_snapshot_size", "qe_snapshot", "qe_restore",
    "qe_launch_overhead",
]
QE_DEBUG_FAIL_DEVICE_ALLOC, QE_DEBUG_FAIL_HOST_STORE, QE_DEBUG_EXPIRE_WAIT, QE_DEBUG_VERIFY_PATH = 1, 2, 3, 4
QE_VERIFY_MAX = 16
QE_TIERING_WINDOWS, QE_TIERING_TOKENS = 0, 1
TOK_BF16, TOK_INT4, TOK_INT2, TOK_NQ1, TOK_EVICTED, TOK_ABSENT = 0, 1, 2, 3, 4, 255


class QEConfig(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("n_layers", ctypes.c_int), ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("window", ctypes.c_int),
        ("route_period", ctypes.c_int), ("n_sink", ctypes.c_int), ("n_recent", ctypes.c_int),
        ("max_context", ctypes.c_int), ("cap_mode", ctypes.c_int), ("kf", ctypes.c_int),
        ("kq", ctypes.c_int), ("frac_bf16", ctypes.c_double), ("frac_int2", ctypes.c_double),
        ("budget_frac", ctypes.c_double), ("out_fp32", ctypes.c_int),
        ("tiering", ctypes.c_int), ("frac_int4", ctypes.c_double), ("frac_nq1", ctypes.c_double),
        ("score_window", ctypes.c_int), ("rope_theta", ctypes.c_double), ("int2_slack", ctypes.c_int),
    ]


class QELayerInfo(ctypes.Structure):
    _fields_ = [
        ("length", ctypes.c_int), ("n_windows", ctypes.c_int), ("routed_upto", ctypes.c_int),
        ("n_full", ctypes.c_int), ("n_quant", ctypes.c_int), ("n_pinned", ctypes.c_int),
        ("kf", ctypes.c_int), ("kq", ctypes.c_int), ("max_windows", ctypes.c_int),
        ("units", ctypes.c_int), ("attn_bytes", ctypes.c_double),
    ]


class QERouteStats(ctypes.Structure):
    _fields_ = [("routes", ctypes.c_longlong), ("first_packs", ctypes.c_longlong),
                ("ledger_reuses", ctypes.c_longlong), ("promotions", ctypes.c_longlong),
                ("evictions", ctypes.c_longlong), ("bf16_reclaims", ctypes.c_longlong),
                ("int2_reclaims", ctypes.c_longlong), ("ledger_writes", ctypes.c_longlong)]


class QERouteDiag(ctypes.Structure):
    """One unit's record of a layer's latest routing event (see qe_route_diag in qe.h)."""
    _fields_ = [(n, ctypes.c_int) for n in ("kf", "kq", "full_old", "full_new", "full_both", "kept_old",
                                             "kept_new", "kept_both", "promotions", "demotions", "evictions")] + \
               [(n, ctypes.c_float) for n in ("full_cut_kept", "full_cut_next", "kept_cut_kept", "kept_cut_next")]


class QEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"qe status {status}: {msg}")
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def load_library() -> ctypes.CDLL:
    """Load libqe.so (raises if it is missing: there is no CPU path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with python -m tiered_quantize_evict_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
    sig = {
        "qe_init": ([ctypes.POINTER(QEConfig), P, ctypes.POINTER(P)], I),
        "qe_destroy": ([P], I),
        "qe_last_error": ([P], ctypes.c_char_p),
        "qe_append": ([P, I, P, P, I, I], I),
        "qe_decode_step": ([P, I, P, P, I], I),
        "qe_route": ([P, I], I),
        "qe_synchronize": ([P], I),
        "qe_get_layer_info": ([P, I, ctypes.POINTER(QELayerInfo)], I),
        "qe_get_tiers": ([P, I, P, S], I),
        "qe_get_scores": ([P, I, P, S], I),
        "qe_set_scores": ([P, I, P, S], I),
        "qe_get_quant_window": ([P, I, I, I, P, P, P, P, P, P], I),
        "qe_get_bf16_window": ([P, I, I, I, P, P], I),
        "qe_get_route_stats": ([P, I, ctypes.POINTER(QERouteStats)], I),
        "qe_set_timing": ([P, I], I),
        "qe_get_timing": ([P, ctypes.POINTER(D), ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(D)], I),
        "qe_launch_overhead": ([P, I, ctypes.POINTER(D)], I),
        "qe_kernel_launches": ([P], ctypes.c_longlong),
        "qe_decode_step_noalloc": ([P, I, P, P], I),
        "qe_get_route_diag": ([P, I, ctypes.POINTER(QERouteDiag), S], I),
        "qe_get_token_tiers": ([P, I, P, S], I),
        "qe_get_token_scores": ([P, I, P, S], I),
        "qe_get_token_counts": ([P, I, P, S], I),
        "qe_get_token": ([P, I, I, I, ctypes.POINTER(I), P, P, P, P, P], I),
        "qe_verify": ([P, I, P, P, P, P, I, I], I),
        "qe_verify_commit": ([P, I, I], I),
        "qe_debug_inject": ([P, I, ctypes.c_longlong], I),
    "qe_snapshot_size": ([P, ctypes.POINTER(ctypes.c_size_t)], I),
    "qe_snapshot": ([P, P, ctypes.c_size_t], I),
    "qe_restore": ([P, P, ctypes.c_size_t], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(x) -> int:
    """Address of a torch tensor or numpy array (no copy)."""
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"]
        return x.ctypes.data
    raise TypeError(type(x))


def _is_host(x) -> bool:
    if isinstance(x, np.ndarray):
        return True
    return not x.is_cuda


def debug_inject(what: int, value: int, cache: Optional["QECache"] = None) -> int:
    """qe_debug_inject: host-side fault injection for tests (returns the status code)."""
    lib = load_library()
    h = cache.h if cache is not None else None
    return int(lib.qe_debug_inject(h, what, value))


class QECache:
    """One cache handle (qe_init .. qe_destroy)."""

    def __init__(self, cfg: QEConfig, stream: int = 0):
        lib = load_library()
        self._lib = lib
        self.cfg = cfg
        h = ctypes.c_void_p()
        st = lib.qe_init(ctypes.byref(cfg), ctypes.c_void_p(stream), ctypes.byref(h))
        if st != QE_OK:
            raise QEError(st, lib.qe_last_error(None).decode())
        self.h = h

    def _check(self, st: int):
        if st != QE_OK:
            raise QEError(st, self._lib.qe_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self._lib.qe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- the path
    def qe_append(self, layer: int, k, v, n_tokens: int):
        flags = QE_HOST_PTRS if _is_host(k) else QE_DEVICE_PTRS
        self._check(self._lib.qe_append(self.h, layer, _ptr(k), _ptr(v), n_tokens, flags))

    def qe_decode_step(self, layer: int, q, out):
        flags = QE_HOST_PTRS if _is_host(q) else QE_DEVICE_PTRS
        self._check(self._lib.qe_decode_step(self.h, layer, _ptr(q), _ptr(out), flags))

    def qe_decode_step_noalloc(self, layer: int, q, out):
        """qe_decode_step without any device allocation (device q/out only; scratch is a static array)."""
        if _is_host(q) or _is_host(out):
            raise ValueError("qe_decode_step_noalloc takes device tensors only")
        self._check(self._lib.qe_decode_step_noalloc(self.h, layer, _ptr(q), _ptr(out)))

    def qe_verify(self, layer: int, q, k, v, out, n_q: int):
        """Speculative verify of n_q drafts: q [n_q][B][Hq][D], k/v [n_q][B][Hkv][D], out [n_q][B][Hq][D]."""
        flags = QE_HOST_PTRS if _is_host(q) else QE_DEVICE_PTRS
        self._check(self._lib.qe_verify(self.h, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(out), n_q, flags))

    def qe_verify_commit(self, layer: int, n_accept: int):
        self._check(self._lib.qe_verify_commit(self.h, layer, n_accept))

    def qe_route(self, layer: int = -1):
        self._check(self._lib.qe_route(self.h, layer))

    def qe_synchronize(self):
        self._check(self._lib.qe_synchronize(self.h))

    # ---------------------------------------------------------------- introspection
    def layer_info(self, layer: int) -> QELayerInfo:
        info = QELayerInfo()
        self._check(self._lib.qe_get_layer_info(self.h, layer, ctypes.byref(info)))
        return info

    def qe_layer_info_sync(self):
        """Resynchronise the host's view of every layer with the device (after graph replays)."""
        for layer in range(self.cfg.n_layers):
            self.layer_info(layer)

    def tiers(self, layer: int) -> np.ndarray:
        info = self.layer_info(layer)
        out = np.zeros((info.units, info.max_windows), np.uint8)
        self._check(self._lib.qe_get_tiers(self.h, layer, out.ctypes.data, out.nbytes))
        return out

    def scores(self, layer: int) -> np.ndarray:
        info = self.layer_info(layer)
        out = np.zeros((info.units, info.max_windows), np.float32)
        self._check(self._lib.qe_get_scores(self.h, layer, out.ctypes.data, out.nbytes))
        return out

    def set_scores(self, layer: int, s: np.ndarray):
        s = np.ascontiguousarray(s, np.float32)
        self._check(self._lib.qe_set_scores(self.h, layer, s.ctypes.data, s.nbytes))

    def quant_window(self, layer: int, unit: int, window: int):
        w, d = self.cfg.window, self.cfg.head_dim
        kc = np.zeros((w, d), np.uint8)
        vc = np.zeros((w, d), np.uint8)
        kz = np.zeros(d, np.float32)
        ks = np.zeros(d, np.float32)
        vz = np.zeros(w, np.float32)
        vs = np.zeros(w, np.float32)
        self._check(self._lib.qe_get_quant_window(self.h, layer, unit, window, kc.ctypes.data, vc.ctypes.data,
                                                  kz.ctypes.data, ks.ctypes.data, vz.ctypes.data, vs.ctypes.data))
        return kc, vc, kz, ks, vz, vs

    def bf16_window(self, layer: int, unit: int, window: int):
        w, d = self.cfg.window, self.cfg.head_dim
        k = np.zeros((w, d), np.uint16)
        v = np.zeros((w, d), np.uint16)
        self._check(self._lib.qe_get_bf16_window(self.h, layer, unit, window, k.ctypes.data, v.ctypes.data))
        return k, v

    def route_stats(self, layer: int = -1) -> QERouteStats:
        s = QERouteStats()
        self._check(self._lib.qe_get_route_stats(self.h, layer, ctypes.byref(s)))
        return s

    def route_diag(self, layer: int):
        """Records of the layer's latest routing event, one per unit."""
        units = self.cfg.batch * self.cfg.n_kv_heads
        arr = (QERouteDiag * units)()
        self._check(self._lib.qe_get_route_diag(self.h, layer, arr, units))
        return list(arr)

    # ---------------------------------------------------------------- five-tier mode
    def token_tiers(self, layer: int) -> np.ndarray:
        """[units][max_context] uint8 tier of every position (TOK_*)."""
        out = np.zeros((self.cfg.batch * self.cfg.n_kv_heads, self.cfg.max_context), np.uint8)
        self._check(self._lib.qe_get_token_tiers(self.h, layer, out.ctypes.data, out.nbytes))
        return out

    def token_scores(self, layer: int) -> np.ndarray:
        out = np.zeros((self.cfg.batch * self.cfg.n_kv_heads, self.cfg.max_context), np.float32)
        self._check(self._lib.qe_get_token_scores(self.h, layer, out.ctypes.data, out.nbytes))
        return out

    def token_counts(self, layer: int) -> np.ndarray:
        """[units][5]: ranked BF16, INT4, INT2, 1-bit, BF16 tail."""
        out = np.zeros((self.cfg.batch * self.cfg.n_kv_heads, 5), np.int32)
        self._check(self._lib.qe_get_token_counts(self.h, layer, out.ctypes.data, out.nbytes))
        return out

    def token(self, layer: int, unit: int, pos: int):
        """(tier, k_bf16 bits, v_bf16 bits, k_codes, v_codes, params[4]) of one position."""
        d = self.cfg.head_dim
        tier = ctypes.c_int()
        kb, vb = np.zeros(d, np.uint16), np.zeros(d, np.uint16)
        kc, vc = np.zeros(d, np.uint8), np.zeros(d, np.uint8)
        par = np.zeros(4, np.float32)
        self._check(self._lib.qe_get_token(self.h, layer, unit, pos, ctypes.byref(tier), kb.ctypes.data, vb.ctypes.data,
                                           kc.ctypes.data, vc.ctypes.data, par.ctypes.data))
        return tier.value, kb, vb, kc, vc, par

    def snapshot(self) -> np.ndarray:
        """qe_snapshot: the handle's whole state as a host byte array (synchronous)."""
        n = ctypes.c_size_t()
        self._check(self._lib.qe_snapshot_size(self.h, ctypes.byref(n)))
        buf = np.empty(n.value, np.uint8)
        self._check(self._lib.qe_snapshot(self.h, buf.ctypes.data, n.value))
        return buf

    def restore(self, snap: np.ndarray):
        """qe_restore: replace the handle's state with a snapshot of a same-config handle."""
        snap = np.ascontiguousarray(snap, dtype=np.uint8)
        self._check(self._lib.qe_restore(self.h, snap.ctypes.data, snap.nbytes))

    def set_timing(self, enable: bool):
        self._check(self._lib.qe_set_timing(self.h, 1 if enable else 0))

    def timing(self):
        ms, n, b = ctypes.c_double(), ctypes.c_longlong(), ctypes.c_double()
        self._check(self._lib.qe_get_timing(self.h, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(b)))
        return ms.value, n.value, b.value

    def kernel_launches(self) -> int:
        return int(self._lib.qe_kernel_launches(self.h))

    def launch_overhead(self, n: int = 100) -> float:
        """qe_launch_overhead: mean event time (us) of an empty launch shaped like the attention's."""
        us = ctypes.c_double()
        self._check(self._lib.qe_launch_overhead(self.h, int(n), ctypes.byref(us)))
        return us.value


def config_from_workload(wl, out_fp32: bool = True, max_context: Optional[int] = None,
                         n_layers: Optional[int] = None, batch: Optional[int] = None) -> QEConfig:
    """QEConfig for a ``qe_inputs.Workload`` (duck-typed: any object with the same fields)."""
    return QEConfig(
        batch=batch or wl.batch, n_layers=n_layers or wl.n_layers, n_q_heads=wl.n_q_heads,
        n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim, window=wl.window,
        route_period=wl.route_period, n_sink=wl.n_sink, n_recent=wl.n_recent,
        max_context=max_context or wl.max_context, cap_mode=wl.cap_mode, kf=wl.kf, kq=wl.kq,
        frac_bf16=wl.frac_bf16, frac_int2=wl.frac_int2, budget_frac=wl.budget_frac,
        out_fp32=1 if out_fp32 else 0,
        tiering=QE_TIERING_TOKENS if getattr(wl, "tiering", "windows") == "tokens" else QE_TIERING_WINDOWS,
        frac_int4=getattr(wl, "frac_int4", 0.0), frac_nq1=getattr(wl, "frac_nq1", 0.0),
        score_window=getattr(wl, "score_window", 0), rope_theta=getattr(wl, "rope_theta", 0.0),
        int2_slack=getattr(wl, "int2_slack", 0))
