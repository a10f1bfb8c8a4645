"""ctypes loader for libpagedkv.so with the signatures of include/pagedkv*.h.

The library is built in-tree (``paged_kv_cache_66_gb300/_build.py``).  Loading
fails loudly when it is missing: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

from . import _build

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
                4: "PA_ERR_DEVICE_CHECK", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_POOL_EXHAUSTED",
                7: "PA_ERR_OVER_RELEASE", 8: "PA_ERR_EXISTS", 9: "PA_ERR_NOT_FOUND"}
DTYPE_IDS = {"f32": 0, "f16": 1, "bf16": 2}

_i32, _i64, _sz, _vp, _f32 = C.c_int, C.c_int64, C.c_size_t, C.c_void_p, C.c_float
_p64 = C.POINTER(C.c_int64)
_p32 = C.POINTER(C.c_int32)

# name -> (restype, argtypes); the exported symbol set of both headers
SIGNATURES = {
    # include/pagedkv.h
    "pa_kv_append": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _i32, _vp]),
    "pa_copy_blocks": (_i32, [C.POINTER(_vp), C.POINTER(_vp), _i32, _vp, _i64, _i64, _sz, _vp]),
    "pa_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_decode": (_i32, [_vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                         _vp, _sz, _i32, _vp]),
    "pa_decode_append": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                _i32, _f32, _i32, _vp, _sz, _i32, _vp]),
    "pa_decode_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                                 _i32, _i32, _vp]),
    "pa_kv_append_fp8": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp]),
    "pa_decode_fp8": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                             _f32, _i32, _vp, _sz, _vp]),
    "pa_prefill": (_i32, [_vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                          _f32, _i32, _vp]),
    "pa_set_decode_kernel": (_i32, [_i32]),
    "pa_set_decode_heads_per_cta": (_i32, [_i32]),
    "pa_selftest_wait_timeout": (_i32, [_i32, _vp]),
    "pa_get_device_error": (_i32, [C.POINTER(C.c_int), _vp]),
    "pa_status_string": (C.c_char_p, [_i32]),
    # include/pagedkv_host.h
    "pa_host_create": (_vp, [_i64, _i32, _p32]),
    "pa_host_destroy": (None, [_vp]),
    "pa_host_seq_create": (_i32, [_vp, _i64]),
    "pa_host_reserve": (_i32, [_vp, _i64, _i64, _p64, _i64, _p64]),
    "pa_host_slots": (_i32, [_vp, _i64, _i64, _i64, _p64]),
    "pa_host_advance": (_i32, [_vp, _i64, _i64]),
    "pa_host_fork": (_i32, [_vp, _i64, _i64]),
    "pa_host_free": (_i32, [_vp, _i64]),
    "pa_host_truncate": (_i32, [_vp, _i64, _i64]),
    "pa_host_length": (_i32, [_vp, _i64, _p64]),
    "pa_host_table": (_i32, [_vp, _i64, _p32, _i64, _p64]),
    "pa_host_num_free": (_i64, [_vp]),
    "pa_host_num_blocks": (_i64, [_vp]),
    "pa_host_refcount": (C.c_int32, [_vp, _i64]),
    "pa_host_batch": (_i32, [_vp, _p64, _i64, _p32, _i64, _p32, _p64]),
    "pa_host_decode_step": (_i32, [_vp, _p64, _i64, _p64, _p64, _i64, _p64, _p32, _i64, _p32, _p64]),
    "pa_host_prefix_attach": (_i32, [_vp, _i64, _p64, _i64, _p64]),
    "pa_host_prefix_remember": (_i32, [_vp, _i64, _p64, _i64]),
    "pa_host_prefix_evict": (_i32, [_vp, _i64]),
    "pa_host_prefix_entries": (_i64, [_vp]),
    "pa_prefix_chain_keys": (_i32, [_p64, _i64, _i32, _vp, _i64, _vp]),
    "pa_host_hprefix_attach": (_i32, [_vp, _i64, _p64, _i64, _vp, _i64, _p64]),
    "pa_host_hprefix_remember": (_i32, [_vp, _i64, _p64, _i64, _vp, _i64]),
    "pa_host_hprefix_evict": (_i32, [_vp, _i64]),
    "pa_host_hprefix_entries": (_i64, [_vp]),
    "pa_host_hprefix_blocks": (_i64, [_vp, _p32, _i64]),
    "pa_host_tprefix_attach": (_i32, [_vp, _i64, _p64, _i64, _p64]),
    "pa_host_tprefix_remember": (_i32, [_vp, _i64, _p64, _i64]),
    "pa_host_tprefix_evict": (_i32, [_vp, _i64]),
    "pa_host_tprefix_nodes": (_i64, [_vp]),
    "pa_host_tprefix_blocks": (_i64, [_vp, _p32, _i64]),
}

_LIB = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> C.CDLL:
    """Load (building first if needed and allowed) and type the library."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path) or not _build.up_to_date():
        if not build_if_missing:
            raise RuntimeError(f"libpagedkv.so is missing at {path}; run paged_kv_cache_66_gb300._build.build()")
        _build.build()
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}" if what else STATUS_NAMES.get(status, status))


def check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedKVError(status, what)
