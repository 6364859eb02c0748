"""ctypes loader for libmuon_ns.so (the C ABI declared in include/muon_ns.h).

The library is built in-tree by newton_schulz_07_gb300.build; there is no
fallback: if it is missing, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmuon_ns.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_ALIGNMENT = 2
ERR_UNSUPPORTED_DEVICE = 3
ERR_WORKSPACE = 4
ERR_CUDA = 5
ERR_TIMEOUT = 6

DEVERR_WAIT_TIMEOUT = 1  # bit of the device error word
HALF = 1  # MUON_NS_HALF: per-step storage of A and B as whole calls keep them

WS_TOTAL, WS_ERROR, WS_NORMS, WS_X, WS_GRAM, WS_POLY, WS_DIAG = range(7)

_c_int, _c_ll, _c_sz, _c_f, _vp = ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
_pf = ctypes.POINTER(ctypes.c_float)
_pi = ctypes.POINTER(ctypes.c_int)
_psz = ctypes.POINTER(ctypes.c_size_t)

class MuonNSStack(ctypes.Structure):
    """muon_ns_stack of include/muon_ns.h."""
    _fields_ = [("G", ctypes.c_void_p), ("out", ctypes.c_void_p), ("batch", ctypes.c_int),
                ("rows", ctypes.c_int), ("cols", ctypes.c_int)]


_pst = ctypes.POINTER(MuonNSStack)


class MuonStepHparams(ctypes.Structure):
    """muon_step_hparams of include/muon_ns.h."""
    _fields_ = [("lr", ctypes.c_float), ("momentum", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("scale", ctypes.c_float), ("nesterov", ctypes.c_int)]


_php = ctypes.POINTER(MuonStepHparams)


class MuonStepStack(ctypes.Structure):
    """muon_step_stack of include/muon_ns.h."""
    _fields_ = [("W", ctypes.c_void_p), ("M", ctypes.c_void_p), ("G", ctypes.c_void_p), ("batch", ctypes.c_int),
                ("rows", ctypes.c_int), ("cols", ctypes.c_int), ("hp", MuonStepHparams)]


_pss = ctypes.POINTER(MuonStepStack)

# name -> (restype, argtypes); the exported C ABI, in header order.
SIGNATURES = {
    "muon_ns_version": (ctypes.c_char_p, []),
    "muon_ns_status_string": (ctypes.c_char_p, [_c_int]),
    "muon_ns_device_supported": (_c_int, [_c_int]),
    "muon_ns_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _psz]),
    "muon_ns_workspace_region": (_c_int, [_c_int, _c_int, _c_int, _c_int, _psz, _psz]),
    "muon_ns_ws": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _pf, _c_f, _vp, _c_sz, _vp]),
    "muon_ns": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _pf, _c_f, _vp]),
    "muon_ns_f32_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _psz]),
    "muon_ns_f32_workspace_region": (_c_int, [_c_int, _c_int, _c_int, _c_int, _psz, _psz]),
    "muon_ns_ws_f32": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _pf, _c_f, _vp, _c_sz, _vp]),
    "muon_ns_grouped_workspace_size": (_c_int, [_pst, _c_int, _psz]),
    "muon_ns_grouped": (_c_int, [_pst, _c_int, _c_int, _pf, _c_f, _vp, _c_sz, _vp]),
    "muon_ns_host_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _c_int, _psz]),
    "muon_ns_host_chunk": (_c_int, [_c_int, _c_int, _c_int, _c_int]),
    "muon_ns_host_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _c_int]),
    "muon_ns_host": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _pf, _c_f, _c_int, _vp, _c_sz, _vp]),
    "muon_ns_read_error": (_c_int, [_vp, _pi, _c_int, _vp]),
    "muon_ns_check": (_c_int, [_vp, _vp, _vp]),
    "muon_ns_cached_error": (_c_int, [_c_int, _pi]),
    "muon_ns_set_wait_budget": (_c_int, [_c_ll]),
    "muon_ns_inject_stall": (_c_int, [_c_int]),
    "muon_ns_normalize": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_f, _vp, _c_sz, _vp]),
    "muon_ns_normalize_static": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_f, _vp]),
    "muon_ns_gram": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _c_f, _vp, _vp]),
    "muon_ns_poly": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_f, _c_f, _vp, _vp]),
    "muon_ns_update": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_f, _vp, _c_f, _vp, _vp]),
    "muon_ns_gram_ex": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _c_f, _c_int, _vp, _vp]),
    "muon_ns_poly_ex": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_f, _c_f, _c_int, _vp, _vp]),
    "muon_ns_update_ex": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_f, _vp, _c_f, _c_int, _vp, _vp]),
    "muon_step_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _psz]),
    "muon_step_ws": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _php, _c_int, _pf, _c_f, _vp, _c_sz, _vp]),
    "muon_momentum": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_f, _c_int, _vp, _c_sz, _vp]),
    "muon_apply": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _php, _vp]),
    "muon_step_grouped_workspace_size": (_c_int, [_pss, _c_int, _psz]),
    "muon_step_grouped": (_c_int, [_pss, _c_int, _c_int, _pf, _c_f, _vp, _c_sz, _vp]),
    "muon_step_launches": (_c_int, [_c_int]),
    "muon_ns_launches_per_call": (_c_int, [_c_int]),
    "muon_ns_tile_count": (_c_ll, [_c_int, _c_int, _c_int, _c_int]),
    "muon_ns_tile_coords": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_ll, _pi, _pi, _pi]),
}

_lock = threading.Lock()
_lib = None


class MuonNSError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().muon_ns_status_string(status).decode()
        super().__init__(f"{where}: status {status} ({msg})")


def lib() -> ctypes.CDLL:
    """The loaded library (loads it on first use; raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m newton_schulz_07_gb300.build` "
                    "(there is no fallback implementation)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def check(status: int, where: str) -> None:
    if status != OK:
        raise MuonNSError(status, where)
