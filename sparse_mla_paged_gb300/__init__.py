"""GB300-native selected-index (DSA) NoPE MLA paged decode.

The decode runs in hand-written sm_103a CUDA kernels behind the C-ABI library
``libdsa_mla.so`` (declared in ``include/dsa_mla.h``). This package holds the thin Python
binding of that library (``api``), the ctypes loader (``_lib``), the in-tree build
(``build``) and the seeded synthetic workloads (``workloads``). The binding never falls
back to anything else: if the CUDA library is missing, every call raises.
"""
from __future__ import annotations

import importlib

__all__ = ["api", "workloads", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
