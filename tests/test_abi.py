"""The C-ABI library builds, loads and exports every entry point qe.h declares (no GPU needed)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qe.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(qe_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import tiered_quantize_evict_gb300 as qe
    if not os.path.exists(qe.LIB_PATH):
        from tiered_quantize_evict_gb300.build import build_library
        build_library()
    return qe.load_library()


def test_header_declarations_are_parsed():
    names = _declared()
    for must in ("qe_init", "qe_append", "qe_decode_step", "qe_route", "qe_destroy"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    import tiered_quantize_evict_gb300 as qe
    names = _declared()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(qe.EXPORTED) == names


def test_init_reports_errors_without_crashing(lib):
    import tiered_quantize_evict_gb300 as qe
    import torch
    cfg = qe.QEConfig(batch=1, n_layers=1, n_q_heads=4, n_kv_heads=1, head_dim=96, window=16,
                      route_period=8, n_sink=4, n_recent=16, max_context=64, cap_mode=0, kf=1, kq=1)
    h = ctypes.c_void_p()
    st = lib.qe_init(ctypes.byref(cfg), None, ctypes.byref(h))
    assert st == qe.QE_ERR_INVALID_ARG and b"head_dim" in lib.qe_last_error(None)
    cfg.head_dim = 64
    cfg.int2_slack = -2
    st = lib.qe_init(ctypes.byref(cfg), None, ctypes.byref(h))
    assert st == qe.QE_ERR_INVALID_ARG and b"int2_slack" in lib.qe_last_error(None)
    cfg.int2_slack = 0
    if not torch.cuda.is_available():
        cfg.head_dim = 64
        st = lib.qe_init(ctypes.byref(cfg), None, ctypes.byref(h))
        assert st == qe.QE_ERR_CUDA and lib.qe_last_error(None)
    assert lib.qe_append(None, 0, None, None, 1, 0) == qe.QE_ERR_INVALID_ARG


def test_debug_inject_validates_its_arguments(lib):
    """qe_debug_inject acts on host state only; its argument checks need no GPU."""
    import tiered_quantize_evict_gb300 as qe
    assert lib.qe_debug_inject(None, qe.QE_DEBUG_EXPIRE_WAIT, 1) == qe.QE_ERR_INVALID_ARG   # needs a handle
    assert lib.qe_debug_inject(None, qe.QE_DEBUG_VERIFY_PATH, 1) == qe.QE_ERR_INVALID_ARG   # needs a handle
    assert lib.qe_debug_inject(None, 99, 1) == qe.QE_ERR_INVALID_ARG
    assert lib.qe_debug_inject(None, qe.QE_DEBUG_FAIL_DEVICE_ALLOC, -1) == qe.QE_ERR_INVALID_ARG
    assert lib.qe_debug_inject(None, qe.QE_DEBUG_FAIL_DEVICE_ALLOC, 0) == qe.QE_OK
    assert lib.qe_debug_inject(None, qe.QE_DEBUG_FAIL_HOST_STORE, 0) == qe.QE_OK
