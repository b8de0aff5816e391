"""ctypes binding of libq3kv.so: symbol prototypes and error mapping only.

Every entry point keeps the C name and argument order of ``include/q3kv.h``.
There is no fallback: if the library is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_int32 = ctypes.c_int32
c_int64 = ctypes.c_int64
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p
P_int32 = ctypes.POINTER(ctypes.c_int32)

Q3KV_OK = 0
Q3KV_ERR_INVALID_ARG = -1
Q3KV_ERR_UNSUPPORTED = -2
Q3KV_ERR_OUT_OF_PAGES = -3
Q3KV_ERR_WORKSPACE_TOO_SMALL = -4
Q3KV_ERR_CUDA = -5
Q3KV_ERR_SLOT_RANGE = -6
Q3KV_ERR_HOST_MEMORY = -7

Q3KV_STATUS_NONFINITE_INPUT = 1
Q3KV_STATUS_SCALE_OVERFLOW = 2
Q3KV_STATUS_BAD_PAGE = 4
Q3KV_STATUS_BAD_LENGTH = 8
Q3KV_STATUS_TIMEOUT = 16
Q3KV_STATUS_RANGE = 32

Q3KV_F32 = 0
Q3KV_BF16 = 1

Q3KV_IMPL_AUTO = 0
Q3KV_IMPL_FMA = 1
Q3KV_IMPL_MMA = 2


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_layers", c_int32), ("num_kv_heads", c_int32), ("num_q_heads", c_int32),
                ("head_dim", c_int32), ("page_size", c_int32), ("num_pages", c_int32)]


P_desc = ctypes.POINTER(CacheDesc)

# name -> (restype, argtypes); mirrors include/q3kv.h
PROTOTYPES = {
    "q3kv_version": (c_int32, []),
    "q3kv_format_version": (c_int32, []),
    "q3kv_strerror": (ctypes.c_char_p, [c_int32]),
    "q3kv_last_cuda_error": (ctypes.c_char_p, []),
    "q3kv_pool_bytes": (c_int32, [P_desc, ctypes.POINTER(c_size_t)]),
    "q3kv_allocator_create": (c_int32, [c_int32, c_int32, c_int32, ctypes.POINTER(c_void_p)]),
    "q3kv_allocator_destroy": (None, [c_void_p]),
    "q3kv_alloc_pages": (c_int32, [c_void_p, c_int32, c_int64, P_int32, P_int32]),
    "q3kv_free_slot": (c_int32, [c_void_p, c_int32]),
    "q3kv_free_pages": (c_int32, [c_void_p, P_int32]),
    "q3kv_append": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                              c_int32, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_void_p]),
    "q3kv_workspace_bytes": (c_int32, [P_desc, c_int32, c_int64, c_int32, c_int32, c_int32,
                                       ctypes.POINTER(c_size_t)]),
    "q3kv_verify_attn": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                   c_int32, c_int64, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                                   c_int32, c_int32, c_void_p, c_size_t, c_void_p]),
    "q3kv_verify_attn_noalloc": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                           c_void_p, c_int32, c_int64, c_int32, c_int32, c_void_p, c_int32,
                                           c_void_p, c_int32, c_int32, c_void_p]),
    "q3kv_prefill_workspace_bytes": (c_int32, [P_desc, c_int32, c_int64, c_int32, c_int32, c_int32,
                                               ctypes.POINTER(c_size_t)]),
    "q3kv_prefill_attn": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                    c_int32, c_int64, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                                    c_int32, c_int32, c_void_p, c_size_t, c_void_p]),
    "q3kv_t5k_pool_bytes": (c_int32, [P_desc, ctypes.POINTER(c_size_t)]),
    "q3kv_t5k_append": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                  c_int32, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_void_p]),
    "q3kv_t5k_verify_attn": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                       c_void_p, c_int32, c_int64, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                                       c_int32, c_int32, c_void_p, c_size_t, c_void_p]),
    "q3kv_fp8_pool_bytes": (c_int32, [P_desc, ctypes.POINTER(c_size_t)]),
    "q3kv_fp8_append": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                  c_int32, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_void_p]),
    "q3kv_fp8_verify_attn": (c_int32, [c_void_p, P_desc, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                       c_void_p, c_int32, c_int64, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                                       c_int32, c_int32, c_void_p, c_size_t, c_void_p]),
    "q3kv_accept_workspace_bytes": (c_int32, [c_int32, c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "q3kv_accept_greedy": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                     c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, ctypes.c_size_t, c_void_p]),
    "q3kv_accept_sample": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                     c_int32, c_int32, c_int32, c_void_p, ctypes.c_float, c_void_p,
                                     ctypes.c_uint64, c_void_p, c_void_p, c_void_p, c_void_p, ctypes.c_size_t,
                                     c_void_p]),
    "q3kv_accept_sample_nucleus": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                             c_int32, c_int32, c_int32, c_void_p, ctypes.c_float, ctypes.c_float,
                                             c_void_p, ctypes.c_uint64, c_void_p, c_void_p, c_void_p, c_void_p,
                                             ctypes.c_size_t, c_void_p]),
}

Q3KV_NOALLOC_SCRATCH_BYTES = 16 << 20

_LIB = None


class Q3KVError(RuntimeError):
    def __init__(self, code: int, where: str):
        detail = ""
        if code == Q3KV_ERR_CUDA:
            detail = ": " + load().q3kv_last_cuda_error().decode()
        super().__init__(f"{where}: {strerror(code)} ({code}){detail}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libq3kv.so (building it first if asked).  Raises if it cannot be had."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise OSError(f"libq3kv.so not found at {path}; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def strerror(code: int) -> str:
    return load().q3kv_strerror(code).decode()


def check(code: int, where: str) -> None:
    if code != Q3KV_OK:
        raise Q3KVError(code, where)
