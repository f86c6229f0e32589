"""ctypes loader for libfa_gb300.so (the C ABI declared in include/fa.h).

There is no fallback: if the library has not been built, load() raises.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

from .build import LIB_PATH, INCLUDE

_lock = threading.Lock()
_lib = None

STATUS_NAMES = {
    0: "FA_OK",
    1: "FA_ERR_INVALID_ARG",
    2: "FA_ERR_UNSUPPORTED",
    3: "FA_ERR_MISALIGNED",
    4: "FA_ERR_WORKSPACE",
    5: "FA_ERR_LAUNCH",
    6: "FA_ERR_TIMEOUT",
    7: "FA_ERR_CUDA",
}

_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p

_SIGNATURES = {
    "fa_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp]),
    "fa_fwd_gqa": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp]),
    "fa_fwd_splitkv": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                _c_float, _c_int, _vp, ctypes.c_size_t, _vp]),
    "fa_fwd_splitkv_workspace_size": (ctypes.c_size_t, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "fa_bwd_workspace_size": (ctypes.c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "fa_bwd_deterministic": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                      _c_int, _c_float, _vp, ctypes.c_size_t, _vp]),
    "fa_bwd_gqa_deterministic": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                          _c_int, _c_int, _c_int, _c_float, _vp, ctypes.c_size_t, _vp]),
    "fa_bwd_gqa_workspace_size": (ctypes.c_size_t, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "fa_bwd_gqa": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                            _c_int, _c_float, _vp, ctypes.c_size_t, _vp]),
    "fa_bwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                        _c_float, _vp, ctypes.c_size_t, _vp]),
    "fa_bwd_preprocess": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, ctypes.c_size_t, _vp]),
    "fa_bwd_preprocess_stats": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, ctypes.c_size_t, _vp]),
    "fa_bwd_main": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp,
                             ctypes.c_size_t, _vp]),
    "fa_bwd_dkdv": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp,
                             ctypes.c_size_t, _vp]),
    "fa_bwd_dq": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp,
                           ctypes.c_size_t, _vp]),
    "fa_bwd_postprocess": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, ctypes.c_size_t, _vp]),
    "fa_bwd_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                _c_float, _vp]),
    "fa_fwd_bwd_host_device_bytes": (ctypes.c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "fa_fwd_host_device_bytes": (ctypes.c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "fa_fwd_host": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp,
                             ctypes.c_size_t, _vp]),
    "fa_fwd_bwd_host": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                 _c_int, _c_float, _vp, ctypes.c_size_t, _vp]),
    "fa_status_string": (ctypes.c_char_p, [_c_int]),
    "fa_get_device_status": (_c_int, [_vp]),
    "fa_get_device_status_detail": (_c_int, [_vp, _vp]),
    "fa_set_wait_limit_ns": (None, [ctypes.c_ulonglong]),
    "fa_debug_timeout_probe": (_c_int, [ctypes.c_ulonglong, _vp]),
    "fa_debug_skip_arrival": (_c_int, [ctypes.c_uint]),
    "fa_version": (_c_int, []),
}


def header_functions() -> list[str]:
    """Names of the functions include/fa.h declares."""
    text = open(os.path.join(INCLUDE, "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def load():
    """Load the built library (once) and declare every C signature."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m exact_softmax_attention_fa_gb300.build` "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        detail = ""
        if _lib is not None:
            s = _lib.fa_status_string(status)
            detail = s.decode() if s else ""
        super().__init__(f"{fn} returned {name}: {detail}")


def check(fn: str, status: int) -> None:
    if status != 0:
        raise FAError(fn, status)
