"""ctypes declarations of the C ABI in include/moe_reorder.h.

Loading fails loudly when libmoe_reorder.so is missing: there is no CPU or
PyTorch fallback for any operation of this package. With USC_CHECKED=1 in the
environment the bounds-checked build (libmoe_reorder_checked.so, built with
-DMR_CHECKED) is loaded instead.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_U64 = ctypes.c_uint64
_U32 = ctypes.c_uint32
_PI64 = ctypes.POINTER(ctypes.c_int64)
_PU64 = ctypes.POINTER(ctypes.c_uint64)

# name -> (restype, argtypes); every function declared in include/moe_reorder.h
SIGNATURES = {
    "ffnwb_batching_get_workspace_size": (_I32, [_I64, _PI64, _I64, _I64, _I64, _PU64]),
    "ffnwb_batching": (_I32, [_P, _I32, _P, _I64, _P, _I64, _P, _P, _P, _I64, _PI64, _I64, _I64,
                              _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _U64, _P]),
    "ffnwb_batching_ex": (_I32, [_P, _I32, _P, _I64, _P, _I64, _P, _P, _P, _I64, _PI64, _I64, _I64,
                                 _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _U32, _P, _U64, _P]),
    "ffnwb_batching_context_get_workspace_size": (_I32, [_I64, _PI64, _I64, _I64, _I64, _PU64]),
    "ffnwb_batching_context": (_I32, [_P, _I64, _PI64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P,
                                      _P, _P, _P, _P, _P, _U64, _P]),
    "ffnwb_batching_context_ex": (_I32, [_P, _I64, _PI64, _I64, _I64, _I64, _I64, _P, _P, _P, _P,
                                         _P, _P, _P, _P, _P, _U32, _P, _U64, _P]),
    "ffnwb_batching_noalloc": (_I32, [_P, _I32, _P, _I64, _P, _I64, _P, _P, _P, _I64, _PI64, _I64,
                                      _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_unpermute_get_workspace_size": (_I32, [_I64, _I64, _I32, _I64, _I32, _I32, _I64, _I64,
                                                _I32, _PI64, _PU64]),
    "moe_unpermute": (_I32, [_P, _P, _P, _P, _I64, _I64, _I32, _I64, _I32, _I64, _I64, _I32, _PI64,
                             _P, _P, _P, _P, _P, _U64, _P]),
    "moe_permute_get_workspace_size": (_I32, [_I64, _I64, _I32, _I64, _I64, _I32, _I64, _PU64]),
    "moe_permute": (_I32, [_P, _P, _I64, _I64, _I32, _I64, _I64, _I32, _I64, _P, _P, _P, _P, _U64,
                           _P]),
    "moe_update_expert": (_I32, [_P, _I32, _P, _P, _I32, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                 _I64, _PI64, _P, _P, _P]),
    "mr_status_string": (ctypes.c_char_p, [_I32]),
    "mr_version": (_I32, []),
    "mr_profile_set_events": (_I32, [ctypes.POINTER(_P), _I32]),
    "mr_checked_errors": (_I32, [ctypes.POINTER(_U32), ctypes.POINTER(_U32), _I32]),
}


def checked_requested() -> bool:
    return os.environ.get("USC_CHECKED", "") == "1"

_lib = None


class LibraryMissing(ImportError):
    pass


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded library (loaded once)."""
    global _lib
    if _lib is None:
        p = path or (_build.CHECKED_LIB_PATH if checked_requested() else _build.LIB_PATH)
        if not os.path.exists(p):
            raise LibraryMissing(
                f"{p} is not built; run unpermute_stable_counting_gb300._build.build_library() "
                "(or __graft_entry__.build()) first")
        L = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def checked_errors(reset: bool = True):
    """(failures, first site) of the bounds checks of a checked build, or None
    for a regular build."""
    f, s = _U32(0), _U32(0)
    st = lib().mr_checked_errors(ctypes.byref(f), ctypes.byref(s), 1 if reset else 0)
    if st == 561003:  # MR_ERR_UNSUPPORTED: a regular build
        return None
    if st != 0:
        raise RuntimeError(f"mr_checked_errors failed with status {st}")
    return int(f.value), int(s.value)


def int64_array(values) -> ctypes.Array:
    arr = (ctypes.c_int64 * len(values))(*[int(v) for v in values])
    return arr
