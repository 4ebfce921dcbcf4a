"""ctypes loader for libdsa_mla.so (the C ABI in include/dsa_mla.h).

There is no fallback: if the library is missing or does not load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa_mla.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dsa_mla.h")

STATUS = {
    0: "DSA_OK",
    1: "DSA_ERR_INVALID_ARGUMENT",
    2: "DSA_ERR_UNSUPPORTED",
    3: "DSA_ERR_WORKSPACE",
    4: "DSA_ERR_CUDA",
    5: "DSA_ERR_NO_KERNEL",
    6: "DSA_ERR_DEVICE_BOUNDS",
    7: "DSA_ERR_TIMEOUT",
}
DSA_OK = 0

_P, _I32, _I64, _F32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class DecodeOptions(ctypes.Structure):
    """dsa_decode_options (include/dsa_mla.h)."""
    _fields_ = [("num_ctas", ctypes.c_int32), ("tile_tokens", ctypes.c_int32), ("gather_mode", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("wait_limit_ns", ctypes.c_uint64),
                ("ev_begin", ctypes.c_void_p), ("ev_end", ctypes.c_void_p)]


_DECODE_ARGS = [_P, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _F32, _F32, _F32, _P]
SIGNATURES = {
    "dsa_abi_version": ([], _I32),
    "dsa_status_string": ([_I32], ctypes.c_char_p),
    "dsa_mla_decode": (_DECODE_ARGS + [_P], _I32),
    "dsa_mla_decode_k": (_DECODE_ARGS + [_P], _I32),
    "dsa_mla_decode_static": (_DECODE_ARGS + [_P], _I32),
    "dsa_mla_decode_workspace_bytes": ([_I32, _I32, _I32, _I32, _I32], _SZ),
    "dsa_mla_decode_grid": ([_I32, _I32, _I32, _I32, _I32], _I32),
    "dsa_mla_decode_ws": (_DECODE_ARGS + [_I32, _P, _SZ, ctypes.POINTER(DecodeOptions), _P], _I32),
    "dsa_mla_decode_host_workspace_bytes": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32], _SZ),
    "dsa_mla_decode_host": ([_P, _P, _P, _P, _I32, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _F32,
                             _F32, _F32, _P, _I32, _P, _SZ, _I32, _P], _I32),
    "dsa_resolve_indices": ([_P, _P, _I32, _I32, _P, _P, _P], _I32),
    "dsa_latent_write": ([_P, _P, _P, _I32, _F32, _F32, _I32, _I64, _P, _P], _I32),
    "dsa_select_pools": ([_P, _P, _I32, _I32, _I32, _I32, _P, _P], _I32),
    "dsa_absorb_q": ([_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P], _I32),
    "dsa_absorb_o": ([_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P], _I32),
    "dsa_read_device_status": ([_P, _P, _P], _I32),
    "dsa_last_device_status": ([_P, _P], _I32),
    "dsa_static_device_status": ([_P, _P], _I32),
}

_lock = threading.Lock()
_lib = None


class DsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def load(path: str = LIB_PATH):
    """Load and declare the library (raises if it is missing: there is no other path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libdsa_mla.so not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def check(status: int, what: str) -> None:
    if status != DSA_OK:
        raise DsaError(status, what)
