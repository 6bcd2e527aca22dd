"""ctypes loader for ``libfa_gb300.so`` with the C signatures of ``include/fa.h``.

There is no fallback: if the library has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")
# the same library with device-side index checks (-DFA_DEBUG)
DEBUG_LIB_PATH = os.path.join(_HERE, "libfa_gb300_debug.so")

FA_OK = 0
FA_ERR_NULLPTR = 1
FA_ERR_PARAM_INVALID = 2
FA_ERR_UNSUPPORTED = 3
FA_ERR_WORKSPACE_TOO_SMALL = 4
FA_ERR_RUNTIME = 5
FA_ERR_DEVICE_TIMEOUT = 6
FA_ERR_DEVICE_CHECK = 7

FA_LAYOUT_BNSD = 0
FA_LAYOUT_BSND = 1
FA_MASK_NONE = 0
FA_MASK_CAUSAL = 3
FA_MASK_WINDOW = 4
FA_LAYOUT_PA_BBND = 2
FA_LAYOUT_PA_BNBD = 3
FA_KEY_MASK_B11S = 0
FA_KEY_MASK_BN1S = 1
FA_KEY_MASK_1N1S = 2

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t

# name -> (restype, argtypes), exactly the declarations of include/fa.h
SIGNATURES = {
    "fa_abi_version": (ctypes.c_int, []),
    "fa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_forward_workspace_size": (_sz, [_i64] * 6),
    "fa_forward": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _i64, _i64, _i64, _i64,
                                  _i64, _i64, ctypes.c_float, ctypes.c_int, _vp, _vp, _vp, _sz,
                                  _vp]),
    "fa_forward_varlen_workspace_size": (_sz, [_i64] * 6),
    "fa_forward_varlen": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _i64, _i64, _i64,
                                         _i64, ctypes.c_float, _vp, _vp, _vp, _sz, _vp]),
    "fa_forward_varlen_window": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                                _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _sz,
                                                _vp]),
    "fa_forward_varlen_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                            _i64, _i64, _i64, _i64, ctypes.c_float, _vp, _vp,
                                            _vp, _sz, _vp]),
    "fa_forward_window": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _vp, _vp, _i64, _i64, _i64,
                                         _i64, _i64, _i64, ctypes.c_float, ctypes.c_int, _vp,
                                         _vp, _vp, _sz, _vp]),
    "fa_forward_paged": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp, _i64, _i64, _i64,
                                        ctypes.c_int, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                        _i64, ctypes.c_float, ctypes.c_int, _vp, _vp, _vp, _sz,
                                        _vp]),
    "fa_decode_paged": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp, _i64, _i64, _i64, _vp,
                                       _vp, _i64, _i64, _i64, _i64, ctypes.c_float, ctypes.c_int,
                                       _vp, _vp, _vp, _sz, _vp]),
    "fa_decode_workspace_size": (_sz, [_i64] * 5 + [ctypes.c_int]),
    "fa_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                 ctypes.c_float, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _sz,
                                 _vp]),
    "fa_decode_masked": (ctypes.c_int, [_vp, _vp, _vp, _vp, ctypes.c_int, _vp, _i64, _i64, _i64,
                                        _i64, _i64, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                        _vp, _vp, _vp, _sz, _vp]),
    "fa_decode_plan": (ctypes.c_int, [_i64, _i64, _i64, _i64, _i64, _vp, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(_i64), ctypes.POINTER(_i64),
                                      ctypes.POINTER(_i64)]),
    "fa_workspace_status": (ctypes.c_int, [_vp, _vp]),
    "fa_selftest_wait_timeout": (ctypes.c_int, [_vp, ctypes.c_uint64, _vp]),
    "fa_decode_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                         ctypes.c_float, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                         _vp]),
    "fa_decode_noalloc_status": (ctypes.c_int, [_vp]),
    "fa_set_wait_timeout_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "fa_set_main_kernel_events": (None, [_vp, _vp]),
    "fa_kernel_launch_count": (ctypes.c_uint64, []),
}

_lock = threading.Lock()
_lib = None
_debug_lib = None


def _open(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load_debug() -> ctypes.CDLL:
    """The debug build (device-side index checks reported as
    FA_ERR_DEVICE_CHECK); same functions as load()'s. Raises if missing."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            _debug_lib = _open(DEBUG_LIB_PATH)
        return _debug_lib


def load() -> ctypes.CDLL:
    """Load the library once; raise if it is missing (no fallback path)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(LIB_PATH)
        return _lib


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().fa_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FaError(status, where)
