"""ctypes loader of libgsort.so: declares every entry point of include/gsort.h.

Loading the library needs no GPU (nothing runs at load time); calling a
compute entry point does.  There is no fallback: if the library is missing
and cannot be built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

c_u32p = ctypes.POINTER(ctypes.c_uint32)
c_i64p = ctypes.POINTER(ctypes.c_int64)


class Options(ctypes.Structure):
    """struct gsort_options."""
    _fields_ = [
        ("spin_limit", ctypes.c_uint32),
        ("stall_tile", ctypes.c_int64),
        ("events", ctypes.POINTER(ctypes.c_void_p)),
        ("num_events", ctypes.c_int),
        ("variant", ctypes.c_int),
    ]


# name -> (restype, argtypes); every symbol that include/gsort.h declares
SIGNATURES = {
    "gsort_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gsort_version": (ctypes.c_int, []),
    "gsort_radix_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int]),
    "gsort_radix_keys": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p]),
    "gsort_radix_pairs": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]),
    "gsort_radix_pairs_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                            ctypes.c_size_t, ctypes.c_void_p,
                                            ctypes.POINTER(Options)]),
    "gsort_radix_sort_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int, ctypes.c_int]),
    "gsort_radix_sort": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p]),
    "gsort_radix_sort_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_size_t, ctypes.c_void_p,
                                           ctypes.POINTER(Options)]),
    "gsort_radix_sort_launch_count": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int]),
    "gsort_digit_histograms": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p]),
    "gsort_compact_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "gsort_compact_positive": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_void_p]),
    "gsort_compact_positive_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int64, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_size_t,
                                                 ctypes.c_void_p, ctypes.POINTER(Options)]),
    "gsort_compact_positive_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p,
                                                      ctypes.c_int64, ctypes.c_void_p,
                                                      ctypes.c_void_p]),
    "gsort_segmented_bitonic": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_void_p]),
    "gsort_segmented_sort_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64,
                                                               ctypes.c_int]),
    "gsort_segmented_sort": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gsort_segmented_sort_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                               ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                               ctypes.POINTER(Options)]),
    "gsort_partition_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "gsort_partition": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gsort_split_sort_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int]),
    "gsort_split_sort": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "gsort_check": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "gsort_radix_num_variants": (ctypes.c_int, []),
    "gsort_radix_variant_name": (ctypes.c_char_p, [ctypes.c_int]),
    "gsort_radix_launch_count": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int]),
}


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load libgsort.so (building it first if it is missing and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"{path} not found; run __graft_entry__.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
