"""ctypes loader for ``libpagedkv.so`` (the C ABI of ``include/pagedkv.h``).

The library is built in-tree by ``paged_kv_cache_264_gb300.build``.  There is no
fallback: if the library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import threading

from . import build as _build

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_CUDA = 3
PKV_ERR_WORKSPACE = 4
PKV_ERR_CAPACITY = 5

PKV_KV_BF16 = 0
PKV_KV_INT8 = 1
PKV_KV_FP8_E4M3 = 2
BLOCK_SIZE = 16

DEVERR_BLOCK_ID = 0x1
DEVERR_CONTEXT_LEN = 0x2
DEVERR_SLOT = 0x4
DEVERR_TIMEOUT = 0x8

# Every function the header declares, with (restype, argtypes).
_vp, _i32, _i64, _sz, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_pi32 = ctypes.POINTER(ctypes.c_int)
_psz = ctypes.POINTER(ctypes.c_size_t)


KERNEL_AUTO = 0
KERNEL_CUDA_CORE = 1
KERNEL_TENSOR_CORE = 2


SCHEDULE_AUTO = 0
SCHEDULE_GRID = 1
SCHEDULE_PERSISTENT = 2


class DecodeOptions(ctypes.Structure):
    _fields_ = [("partition_blocks", ctypes.c_int), ("kernel", ctypes.c_int), ("schedule", ctypes.c_int),
                ("stages", ctypes.c_int), ("blocks_per_stage", ctypes.c_int), ("num_queries", ctypes.c_int),
                ("window", ctypes.c_int), ("reserved", ctypes.c_int * 1)]


SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [_i32]),
    "pkv_last_cuda_error": (ctypes.c_char_p, []),
    "pkv_version": (ctypes.c_char_p, []),
    "pkv_pool_bytes": (_i32, [_i64, _i32, _i32, _i32, _psz, _psz]),
    "pkv_pool_create": (_i32, [_i64, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)]),
    "pkv_pool_destroy": (_i32, [_vp]),
    "pkv_reshape_and_cache": (_i32, [_vp, _vp, _vp, _vp, _i64, _vp]),
    "pkv_decode_workspace_bytes": (_i32, [_vp, _i32, _i32, _i32, ctypes.POINTER(DecodeOptions), _psz]),
    "pkv_decode_plan": (_i32, [_vp, _i32, _i32, _i32, ctypes.POINTER(DecodeOptions), _pi32, _pi32, _pi32,
                               _pi32]),
    "pkv_paged_attention_decode": (_i32, [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "pkv_paged_attention_decode_ex": (_i32, [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _sz,
                                             ctypes.POINTER(DecodeOptions), _vp]),
    "pkv_get_device_error": (_i32, [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]),
    "pkv_launch_count": (ctypes.c_uint64, []),
    "pkv_paged_attention_decode_static_scratch": (_i32, [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _f32,
                                                         _vp, _vp]),
    "pkv_static_scratch_error": (ctypes.c_char_p, []),
    "pkv_copy_blocks": (_i32, [_vp, _vp, _i32, _vp]),
    "pkv_selftest_bounded_wait": (_i32, [ctypes.c_uint64, _vp, _vp, _vp]),
    "pkv_block_manager_create": (_i32, [_i64, _i32, _i32, ctypes.POINTER(_vp)]),
    "pkv_block_manager_destroy": (_i32, [_vp]),
    "pkv_block_manager_add_sequence": (_i32, [_vp, _pi32]),
    "pkv_block_manager_fork": (_i32, [_vp, _i32, _pi32]),
    "pkv_block_manager_free_sequence": (_i32, [_vp, _i32]),
    "pkv_block_manager_append": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _pi32]),
    "pkv_block_manager_truncate": (_i32, [_vp, _i32, _i32]),
    "pkv_block_manager_release_before": (_i32, [_vp, _i32, _i32]),
    "pkv_block_manager_tables": (_i32, [_vp, _vp, _i32, _vp, _vp]),
    "pkv_block_manager_stats": (_i32, [_vp, ctypes.POINTER(ctypes.c_int64), _pi32]),
    "pkv_block_manager_refcount": (ctypes.c_int32, [_vp, ctypes.c_int32]),
}

STATIC_SCRATCH_BYTES = 16 << 20

_LOCK = threading.Lock()
_LIB: ctypes.CDLL | None = None


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        lib = _LIB
        text = lib.pkv_status_string(status).decode() if lib else str(status)
        detail = ""
        if status == PKV_ERR_CUDA and lib is not None:
            detail = ": " + lib.pkv_last_cuda_error().decode()
        super().__init__(f"{what} failed: {text}{detail}")
        self.status = status


def load(path=None) -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _LIB
    with _LOCK:
        if _LIB is not None and path is None:
            return _LIB
        p = path or _build.library_path()
        if not p.exists():
            raise ImportError(
                f"libpagedkv.so not found at {p}; build it with "
                "`python -m paged_kv_cache_264_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(str(p))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _LIB = lib
        return lib


def check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PagedKVError(status, what)
