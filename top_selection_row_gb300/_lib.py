"""ctypes binding of libqrita.so (argument marshalling only).

The shared library must exist: there is no fallback of any kind. Build it
with ``python -m top_selection_row_gb300.build`` or ``__graft_entry__.build()``.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

# Names declared by include/qrita.h, checked by the ABI test.
EXPORTED = (
    "qrita_select",
    "qrita_select_ex",
    "qrita_host_staging_bytes",
    "qrita_select_host",
    "qrita_topk_ids",
    "qrita_candidates",
    "qrita_delta_table",
    "qrita_strerror",
    "qrita_version",
)

_lib = None


def lib() -> ctypes.CDLL:
    """Load libqrita.so once; raise loudly when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libqrita.so is not built ({LIB_PATH}); run __graft_entry__.build() first"
        )
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    L.qrita_select.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp]
    L.qrita_select.restype = i32
    L.qrita_select_ex.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp, u32, vp, vp]
    L.qrita_select_ex.restype = i32
    L.qrita_host_staging_bytes.argtypes = [i32, i64, i64]
    L.qrita_host_staging_bytes.restype = sz
    L.qrita_select_host.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp, sz, vp]
    L.qrita_select_host.restype = i32
    L.qrita_topk_ids.argtypes = [vp, i32, i64, i64, vp, i32, vp, vp, vp]
    L.qrita_topk_ids.restype = i32
    L.qrita_candidates.argtypes = [vp, i32, i64, i64, vp, i32, vp, vp, vp, vp, vp, vp]
    L.qrita_candidates.restype = i32
    L.qrita_delta_table.argtypes = [i32, vp, i32]
    L.qrita_delta_table.restype = i32
    L.qrita_strerror.argtypes = [i32]
    L.qrita_strerror.restype = ctypes.c_char_p
    L.qrita_version.argtypes = []
    L.qrita_version.restype = i32
    _lib = L
    return L
