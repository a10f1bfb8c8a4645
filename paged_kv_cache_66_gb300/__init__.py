"""Paged KV cache for GB300 (sm_103a): PagedAttention decode, KV append and
copy-on-write as CUDA kernels behind a C ABI (libpagedkv.so), a C++ host
block manager, and their Python bindings.

  api      -- pa_kv_append, pa_copy_blocks, pa_decode, pa_decode_workspace_size,
              pa_get_device_error, pa_status_string   (include/pagedkv.h)
  host     -- HostBlockManager                          (include/pagedkv_host.h)
  replay   -- drives a seeded workload through both
"""
from ._lib import PagedKVError, load  # noqa: F401

__all__ = ["PagedKVError", "load"]
