"""Loads libccc.so and declares its C signatures (include/ccc.h).

Raises ImportError with the build command when the library is missing, so a
missing extension can never silently fall back to anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_PATH = os.path.join(_PKG, "libccc.so")
_lock = threading.Lock()
_handle = None

EXPORTS = ("ccc_workspace_size", "ccc_fwd", "ccc_bwd", "ccc_fwd_ex", "ccc_bwd_ex", "ccc_bwd_noalloc",
           "ccc_update", "ccc_update_ex", "ccc_check_status_words", "ccc_check", "ccc_status_string",
           "ccc_last_launch_count")

# Launch option bits of ccc_fwd_ex / ccc_bwd_ex (include/ccc.h).
OPT_OVERLAP_PROLOGUE = 1 << 0

# Size of the fixed scratch array behind ccc_bwd_noalloc (CCC_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 16 << 20


def path() -> str:
    return _PATH


def lib() -> ctypes.CDLL:
    global _handle
    if _handle is not None:
        return _handle
    with _lock:
        if _handle is None:
            if not os.path.exists(_PATH):
                raise ImportError(
                    f"{_PATH} is missing: build it with "
                    "`python -c \"import __graft_entry__ as g; g.build()\"`")
            h = ctypes.CDLL(_PATH)
            P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
            h.ccc_workspace_size.argtypes = [i64, i32, i32, i32]
            h.ccc_workspace_size.restype = sz
            h.ccc_fwd.argtypes = [P, i64, i32, i64, P, i32, i32, P, i32, i32, P, i32, i32, i64, i64, i64,
                                  P, i32, P, P, P, i64, P, P, sz, P]
            h.ccc_fwd.restype = ctypes.c_int
            h.ccc_bwd.argtypes = [P, i64, i32, i64, P, i32, i32, P, i32, i32, P, P, i32, P, P, P, i64, P,
                                  P, i64, P, P, P, P, sz, P]
            h.ccc_bwd.restype = ctypes.c_int
            u32 = ctypes.c_uint32
            h.ccc_fwd_ex.argtypes = h.ccc_fwd.argtypes[:-1] + [u32, P]
            h.ccc_fwd_ex.restype = ctypes.c_int
            h.ccc_bwd_ex.argtypes = h.ccc_bwd.argtypes[:-1] + [u32, P]
            h.ccc_bwd_ex.restype = ctypes.c_int
            h.ccc_bwd_noalloc.argtypes = [P, i64, i32, i64, P, i32, i32, P, i32, i32, P, P, i32, P, P, P,
                                          i64, P, P, i64, P, P, P, P]
            h.ccc_bwd_noalloc.restype = ctypes.c_int
            h.ccc_update.argtypes = [P, i64, i32, i64, P, i32, i32, P, i32, i32, P, i32, i32, i64, i64, i64,
                                     P, i32, P, P, P, i64, P]
            h.ccc_update.restype = ctypes.c_int
            h.ccc_update_ex.argtypes = h.ccc_update.argtypes[:-1] + [ctypes.c_uint32, P]
            h.ccc_update_ex.restype = ctypes.c_int
            h.ccc_check_status_words.argtypes = [i32]
            h.ccc_check_status_words.restype = sz
            h.ccc_check.argtypes = [i64, P, i32, P, i32, P, i32, P, sz, P]
            h.ccc_check.restype = ctypes.c_int
            h.ccc_status_string.argtypes = [ctypes.c_int]
            h.ccc_status_string.restype = ctypes.c_char_p
            h.ccc_last_launch_count.argtypes = []
            h.ccc_last_launch_count.restype = ctypes.c_int
            _handle = h
    return _handle


def status_string(code: int) -> str:
    return lib().ccc_status_string(code).decode()
