"""ctypes loader for libkda.so (the C ABI declared in include/kda.h).

There is no fallback: if the library has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

# Every symbol include/kda.h declares.
EXPORTS = ("kda_decode", "kda_decode_ex", "kda_prefill", "kda_block_tkg", "kda_block_tkg_static",
           "kda_block_tkg_workspace_size", "kda_status_string", "kda_version")

STATUS = {
    0: "KDA_OK", -1: "KDA_ERR_NULL", -2: "KDA_ERR_SHAPE", -3: "KDA_ERR_UNSUPPORTED",
    -4: "KDA_ERR_ENUM", -5: "KDA_ERR_CUDA", -6: "KDA_ERR_ALIGN", -7: "KDA_ERR_VALUE",
    -8: "KDA_ERR_WORKSPACE",
}


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.kda_decode.restype = i
    lib.kda_decode.argtypes = [vp] * 11 + [i, f] + [i] * 7 + [vp, vp]
    lib.kda_prefill.restype = i
    lib.kda_prefill.argtypes = [vp] * 11 + [i, f] + [i] * 7 + [vp, vp]
    lib.kda_decode_ex.restype = i
    lib.kda_decode_ex.argtypes = [vp] * 11 + [i, f, i, i] + [i] * 7 + [vp, vp]
    lib.kda_block_tkg.restype = i
    lib.kda_block_tkg.argtypes = [vp] * 13 + [f] * 4 + [i] * 7 + [vp, ctypes.c_size_t, vp, vp]
    lib.kda_block_tkg_static.restype = i
    lib.kda_block_tkg_static.argtypes = [vp] * 13 + [f] * 4 + [i] * 7 + [vp, vp]
    lib.kda_block_tkg_workspace_size.restype = ctypes.c_size_t
    lib.kda_block_tkg_workspace_size.argtypes = [i] * 7
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [i]
    lib.kda_version.restype = ctypes.c_char_p
    lib.kda_version.argtypes = []
    return lib


def lib_path() -> str:
    return _build.LIB_PATH


_variants: dict = {}


def load_variant(name: str) -> ctypes.CDLL:
    """Load a variant build of the library (see build.VARIANTS), e.g.
    "outgate_swish": the fused block with a swish output gate.  Same symbols
    and signatures as libkda.so.  Raises RuntimeError when it is missing."""
    with _lock:
        if name not in _variants:
            path = _build.VARIANTS[name][0]
            if not os.path.exists(path):
                raise RuntimeError(f"{os.path.basename(path)} not found at {path}: build it with "
                                   "`python -m kda_decode_recurrence_gb300.build`")
            _variants[name] = _declare(ctypes.CDLL(path))
    return _variants[name]


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libkda.so.  Raises RuntimeError when it is missing (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(
                        f"libkda.so not found at {path}: build it with "
                        "`python -m kda_decode_recurrence_gb300.build`")
                _build.build()
            _lib = _declare(ctypes.CDLL(path))
    return _lib
