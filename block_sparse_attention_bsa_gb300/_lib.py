"""ctypes declarations of the libbsa C ABI (include/bsa.h)."""

from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

_lock = threading.Lock()
_lib = None


class BsaTensor(ctypes.Structure):
    _fields_ = [
        ("ptr", ctypes.c_void_p),
        ("B", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("D", ctypes.c_int64),
        ("stride_b", ctypes.c_int64),
        ("stride_s", ctypes.c_int64),
        ("stride_h", ctypes.c_int64),
    ]


STATUS_NAMES = {
    0: "BSA_OK",
    1: "BSA_ERR_INVALID_ARG",
    2: "BSA_ERR_UNSUPPORTED",
    3: "BSA_ERR_WORKSPACE",
    4: "BSA_ERR_CUDA",
    5: "BSA_ERR_INVALID_INDICES",
    6: "BSA_ERR_TIMEOUT",
}

# name -> (restype, argtypes)
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_TP = ctypes.POINTER(BsaTensor)
SIGNATURES = {
    "bsa_version": (_I, []),
    "bsa_get_last_error": (ctypes.c_char_p, []),
    "bsa_select_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "bsa_select": (_I, [_TP, _TP, _I32, _P, _I32, _I32, _P, _I32, _P, _P, _P, _SZ, _P]),
    "bsa_select_rope": (_I, [_TP, _TP, _P, _P, _P, _P, _I32, _P, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P,
                             _SZ, _P]),
    "bsa_select_noalloc": (_I, [_TP, _TP, _I32, _P, _I32, _I32, _P, _I32, _P, _P, _P]),
    "bsa_forward_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "bsa_forward": (_I, [_TP, _TP, _TP, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P, _P,
                         _P, _SZ, _P]),
    "bsa_forward_causal": (_I, [_TP, _TP, _TP, _I32, _I32, ctypes.c_float, _P, _P, _P, _SZ, _P]),
    "bsa_backward_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "bsa_backward": (_I, [_TP, _TP, _TP, _TP, _TP, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float,
                          _P, _P, _P, _P, _SZ, _P]),
    "bsa_validate_indices": (_I, [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _I32, _I32, _P, _P]),
    "bsa_device_status": (_I, [_P]),
    "bsa_debug_wait_probe": (_I, [_I32, ctypes.c_uint64, _P]),
}


def lib_path() -> str:
    return LIB


def load(path: str | None = None):
    """Loads libbsa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB
        if not os.path.exists(p):
            raise RuntimeError(
                f"libbsa.so not found at {p}: build it first "
                "(python -m block_sparse_attention_bsa_gb300.build); there is no fallback path")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib
