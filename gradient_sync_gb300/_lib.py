"""ctypes declarations of libar_gb300.so (the C ABI in include/ar.h)."""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libar_gb300.so")

c_int, c_size_t, c_float, c_void_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
VOIDPP = ctypes.POINTER(c_void_p)
SIZEP = ctypes.POINTER(c_size_t)
INTP = ctypes.POINTER(c_int)


class ArDesc(ctypes.Structure):
    _fields_ = [("n_ranks", c_int), ("count", c_size_t), ("dtype", c_int), ("algo", c_int),
                ("group_size", c_int), ("order", c_int), ("scale", c_float), ("collective", c_int),
                ("sm_budget", c_int), ("kernel", c_int), ("torus_dims", c_int * 3)]


class ArStats(ctypes.Structure):
    _fields_ = [("steps", c_int), ("launches", c_int), ("bytes_sent_per_rank", c_size_t),
                ("hbm_bytes", c_size_t), ("workspace_bytes", c_size_t)]


class ArFabric(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_double), ("bw_local", ctypes.c_double), ("bw_net", ctypes.c_double),
                ("ranks_per_server", c_int), ("in_network", c_int), ("shared_memory", c_int)]


# name -> (restype, argtypes), in the order of include/ar.h
SIGNATURES = {
    "ar_plan": (c_int, [ctypes.POINTER(ArDesc), ctypes.POINTER(c_void_p)]),
    "ar_plan_stats": (c_int, [c_void_p, ctypes.POINTER(ArStats)]),
    "ar_plan_desc": (c_int, [c_void_p, ctypes.POINTER(ArDesc)]),
    "ar_execute": (c_int, [c_void_p, VOIDPP, VOIDPP, c_void_p, c_void_p]),
    "ar_execute_host": (c_int, [c_void_p, VOIDPP, VOIDPP, VOIDPP, c_void_p, c_void_p]),
    "ar_execute_noalloc": (c_int, [c_void_p, VOIDPP, VOIDPP, c_void_p]),
    "ar_bind": (c_int, [c_void_p, VOIDPP, VOIDPP, c_void_p, ctypes.POINTER(c_void_p)]),
    "ar_execute_bound": (c_int, [c_void_p, c_void_p]),
    "ar_bound_destroy": (None, [c_void_p]),
    "ar_plan_destroy": (None, [c_void_p]),
    "ar_plan_predict": (c_int, [c_void_p, ctypes.POINTER(ArFabric), ctypes.POINTER(ctypes.c_double)]),
    "ar_select": (c_int, [ctypes.POINTER(ArDesc), ctypes.POINTER(ArFabric), INTP, INTP,
                          ctypes.POINTER(ctypes.c_double)]),
    "ar_plan_transfers": (c_int, [c_void_p, c_int, INTP, INTP, ctypes.POINTER(ctypes.c_int64), c_int]),
    "ar_bucket_plan": (c_int, [SIZEP, c_int, c_size_t, c_size_t, INTP, INTP]),
    "ar_bucket_pack": (c_int, [c_int, VOIDPP, SIZEP, c_int, c_int, c_int, c_int, VOIDPP, c_void_p]),
    "ar_bucket_unpack": (c_int, [c_int, VOIDPP, c_float, c_int, VOIDPP, SIZEP, c_int, c_int, c_int,
                                 c_void_p]),
    "ar_bucket_allreduce": (c_int, [c_int, VOIDPP, SIZEP, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                    c_void_p]),
    "ar_compress_sizes": (c_int, [c_size_t, c_int, SIZEP, SIZEP]),
    "ar_compress": (c_int, [c_int, c_size_t, c_int, c_int, VOIDPP, VOIDPP, VOIDPP, VOIDPP, c_void_p]),
    "ar_compressed_reduce": (c_int, [c_int, c_size_t, c_int, VOIDPP, VOIDPP, c_float, c_int, VOIDPP, c_void_p]),
    "ar_compressed_allreduce": (c_int, [c_int, c_size_t, c_int, c_int, VOIDPP, VOIDPP, c_float, VOIDPP,
                                        c_void_p]),
    "ar_device_status": (c_int, [c_int]),
    "ar_plan_query": (c_int, [c_void_p]),
    "ar_selftest_wait_timeout": (c_int, [ctypes.c_uint, c_void_p]),
    "ar_selftest_scale_quotient": (c_int, [ctypes.POINTER(ctypes.c_ulonglong)]),
    "ar_status_string": (ctypes.c_char_p, [c_int]),
    "ar_version": (c_int, []),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load the library; fail loudly if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m gradient_sync_gb300.build` "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def ptr_array(ptrs):
    arr = (c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr
