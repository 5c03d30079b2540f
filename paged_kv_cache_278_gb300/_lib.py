"""ctypes loader for libpkv.so (the C ABI declared in include/pkv.h).

The shared library is built in-tree by ``paged_kv_cache_278_gb300.build`` (or
``__graft_entry__.build()``).  There is no fallback: if the library is missing
or fails to load, importing the binding raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

c_int, c_int64, c_size_t, c_float, c_void_p, c_uint64, c_uint = (
    ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint)
c_i32p = ctypes.POINTER(ctypes.c_int32)
c_i64p = ctypes.POINTER(ctypes.c_int64)

# status codes (mirror include/pkv.h)
PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_CUDA = -3
PKV_ERR_OUT_OF_BLOCKS = -4
PKV_ERR_WORKSPACE = -5
PKV_ERR_DEVICE_CHECK = -6

PKV_DEV_OK = 0
PKV_DEV_BAD_BLOCK_ID = 1
PKV_DEV_BAD_CONTEXT = 2
PKV_DEV_BAD_SLOT = 3
PKV_DEV_WAIT_TIMEOUT = 4
PKV_DEV_PREFIX_MISMATCH = 5
PKV_DEV_SMEM_MISALIGNED = 6

PKV_HEAD_DIM = 128
PKV_DEFAULT_PARTITION = 1024
PKV_MAX_PARTITION = 4096
PKV_STEP_OVERLAP = 1
PKV_MAX_QUERY_LEN = 1024
PKV_MAX_STEP_QUERY_LEN = 16
PKV_NOALLOC_SCRATCH_BYTES = 16 << 20

# every symbol include/pkv.h declares: name -> (restype, argtypes)
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [c_int]),
    "pkv_version": (c_int, []),
    "pkv_pool_create": (c_int, [c_int64, c_uint64, ctypes.POINTER(c_void_p)]),
    "pkv_pool_destroy": (None, [c_void_p]),
    "pkv_pool_alloc": (c_int, [c_void_p, c_int, c_i32p]),
    "pkv_pool_share": (c_int, [c_void_p, c_int, c_i32p]),
    "pkv_pool_free": (c_int, [c_void_p, c_int, c_i32p]),
    "pkv_pool_num_free": (c_int64, [c_void_p]),
    "pkv_pool_refcount": (c_int, [c_void_p, ctypes.c_int32]),
    "pkv_pool_reserve": (c_int, [c_void_p, c_i32p, c_int, c_int, c_int, c_int]),
    "pkv_pool_fork": (c_int, [c_void_p, c_i32p, c_i32p, c_int, c_int, c_int]),
    "pkv_pool_prepare_append": (c_int, [c_void_p, c_i32p, c_int, c_int, c_int, c_i32p, c_i32p,
                                        ctypes.POINTER(c_int)]),
    "pkv_pool_free_table": (c_int, [c_void_p, c_i32p, c_int, c_int]),
    "pkv_append_int8k": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                 c_int, c_int64, c_void_p]),
    "pkv_decode_attention_int8k": (c_int, [c_void_p] * 7 + [c_int] * 6 + [c_int64, c_float, c_void_p, c_size_t,
                                                                           c_void_p]),
    "pkv_decode_step_int8k": (c_int, [c_void_p] * 9 + [c_int] * 6 + [c_int64, c_float, c_void_p, c_size_t,
                                                                      c_uint, c_void_p]),
    "pkv_decode_step_partition": (c_int, [c_void_p] * 8 + [c_int] * 6 + [c_int64, c_float, c_int, c_void_p, c_size_t,
                                                                         c_uint, c_void_p]),
    "pkv_decode_multi_workspace_size": (c_size_t, [c_int] * 7),
    "pkv_decode_attention_multi": (c_int, [c_void_p] * 7 + [c_int] * 8 + [c_int64, c_float, c_void_p, c_size_t,
                                                                           c_void_p]),
    "pkv_decode_step_multi": (c_int, [c_void_p] * 9 + [c_int] * 8 + [c_int64, c_float, c_void_p, c_size_t, c_uint,
                                                                      c_void_p]),
    "pkv_pool_swap": (c_int, [c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_i32p, c_i32p]),
    "pkv_copy_blocks_between": (c_int, [c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_int64, c_void_p,
                                        c_void_p, c_int, c_int, c_int, c_int, c_void_p]),
    "pkv_append_int8kv": (c_int, [c_void_p] * 7 + [c_int] * 4 + [c_int64, c_void_p]),
    "pkv_decode_attention_int8kv": (c_int, [c_void_p] * 8 + [c_int] * 6 + [c_int64, c_float, c_void_p, c_size_t,
                                                                            c_void_p]),
    "pkv_decode_step_int8kv": (c_int, [c_void_p] * 10 + [c_int] * 6 + [c_int64, c_float, c_void_p, c_size_t,
                                                                        c_uint, c_void_p]),
    "pkv_append_fp8kv": (c_int, [c_void_p] * 7 + [c_int] * 4 + [c_int64, c_void_p]),
    "pkv_decode_attention_fp8kv": (c_int, [c_void_p] * 8 + [c_int] * 6 + [c_int64, c_float, c_void_p, c_size_t,
                                                                           c_void_p]),
    "pkv_decode_step_fp8kv": (c_int, [c_void_p] * 10 + [c_int] * 6 + [c_int64, c_float, c_void_p, c_size_t,
                                                                       c_uint, c_void_p]),
    "pkv_copy_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int64, c_void_p]),
    "pkv_slot_mapping": (c_int, [c_i64p, c_i32p, c_i32p, c_int, c_int, c_int]),
    "pkv_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                           c_int64, c_void_p]),
    "pkv_decode_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "pkv_decode_attention": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                     c_int, c_int, c_int, c_int, c_int64, c_float, c_void_p, c_size_t,
                                     c_void_p]),
    "pkv_decode_attention_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                             c_int, c_int, c_int, c_int, c_int, c_int64, c_float, c_void_p]),
    "pkv_shared_prefix_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "pkv_decode_attention_shared_prefix": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                   c_int, c_int, c_int, c_int, c_int, c_int, c_int64, c_float,
                                                   c_int, c_void_p, c_size_t, c_void_p]),
    "pkv_decode_step_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "pkv_decode_step": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_int, c_int, c_int, c_int, c_int, c_int, c_int64, c_float, c_int, c_void_p,
                                c_size_t, c_uint, c_void_p]),
    "pkv_decode_partition": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int64, c_float,
                                     c_int, c_int, c_void_p]),
    "pkv_merge": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                          c_void_p]),
    "pkv_get_device_error": (c_int, [c_void_p, ctypes.POINTER(c_int)]),
}


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


_loaded: dict = {}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpkv.so (or another build of the same sources at `path`) once per path, with the
    argument and result types of every declared call; raises if it has not been built."""
    lib = _loaded.get(path)
    if lib is not None:
        return lib
    if not os.path.exists(path):
        raise ImportError(f"libpkv.so is not built ({path}); run `python -m paged_kv_cache_278_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _loaded[path] = lib
    return lib


def status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()


def check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, what)
