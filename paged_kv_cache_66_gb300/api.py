"""Python binding of the device entry points of include/pagedkv.h.

Argument marshalling only: each function checks that the torch tensors it is
given have the layout the C ABI documents, passes their device pointers and
the current CUDA stream, and raises ``PagedKVError`` on a non-OK status.  All
computation happens in the CUDA kernels of libpagedkv.so; there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes as C

import torch

from ._lib import DTYPE_IDS, PagedKVError, check, load

_TORCH_TO_ID = {torch.float32: DTYPE_IDS["f32"], torch.float16: DTYPE_IDS["f16"],
                torch.bfloat16: DTYPE_IDS["bf16"]}

__all__ = ["pa_kv_append", "pa_copy_blocks", "pa_decode_workspace_size", "pa_decode", "pa_decode_noalloc",
           "pa_kv_append_fp8", "pa_decode_fp8", "pa_set_decode_kernel", "pa_decode_append", "pa_get_device_error", "pa_status_string", "PagedKVError"]


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None, dim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {t.dim()}")
    return C.c_void_p(t.data_ptr())


def _dtype_id(t: torch.Tensor) -> int:
    if t.dtype not in _TORCH_TO_ID:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _TORCH_TO_ID[t.dtype]


def pa_kv_append(k, v, k_pool, v_pool, slot_mapping, stream=None) -> None:
    """Scatter k, v [T, Hkv, D] into pools [N, Hkv, b, D] at slot_mapping [T] (int64)."""
    lib = load()
    N, Hkv, b, D = k_pool.shape
    if tuple(v_pool.shape) != tuple(k_pool.shape) or k.shape != v.shape or k.dim() != 3 \
            or k.shape[1:] != (Hkv, D) or slot_mapping.shape != (k.shape[0],):
        raise ValueError("shape mismatch: k, v [T, Hkv, D]; pools [N, Hkv, b, D]; slots [T]")
    dt = k_pool.dtype
    check(lib.pa_kv_append(_dev(k, "k", dt), _dev(v, "v", dt), _dev(k_pool, "k_pool", dt),
                           _dev(v_pool, "v_pool", dt), _dev(slot_mapping, "slot_mapping", torch.int64),
                           k.shape[0], N, Hkv, D, b, _dtype_id(k_pool), _stream(stream)), "pa_kv_append")


def pa_copy_blocks(k_pools, v_pools, pairs, stream=None) -> None:
    """Copy block src -> dst for every (src, dst) row of ``pairs`` ([n, 2] int64 on
    the device) in every layer's K and V pool."""
    lib = load()
    L = len(k_pools)
    if L == 0 or len(v_pools) != L:
        raise ValueError("k_pools and v_pools must be equally long, non-empty lists")
    shape, dt = tuple(k_pools[0].shape), k_pools[0].dtype
    for t in list(k_pools) + list(v_pools):
        if tuple(t.shape) != shape or t.dtype != dt:
            raise ValueError("all pools must share shape and dtype")
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [n, 2]")
    n = pairs.shape[0]
    kp = (C.c_void_p * L)(*[_dev(t, "k_pool").value for t in k_pools])
    vp = (C.c_void_p * L)(*[_dev(t, "v_pool").value for t in v_pools])
    block_bytes = k_pools[0][0].numel() * k_pools[0].element_size()
    pp = _dev(pairs, "pairs", torch.int64) if n > 0 else C.c_void_p(0)
    check(lib.pa_copy_blocks(kp, vp, L, pp, n, shape[0], block_bytes, _stream(stream)), "pa_copy_blocks")


def pa_decode_workspace_size(batch, num_q_heads, head_dim, max_blocks, block_size, partition_tokens=0) -> int:
    return int(load().pa_decode_workspace_size(batch, num_q_heads, head_dim, max_blocks, block_size,
                                               partition_tokens))


def pa_decode(out, q, k_pool, v_pool, block_tables, seq_lens, scale, partition_tokens=0, workspace=None,
              stream=None) -> None:
    """out, q [B, Hq, D]; pools [N, Hkv, b, D]; block_tables [B, max_blocks] int32;
    seq_lens [B] int32; workspace: a uint8 CUDA tensor of at least
    pa_decode_workspace_size(...) bytes (or None when that size is 0)."""
    lib = load()
    B, Hq, D = q.shape
    N, Hkv, b, D2 = k_pool.shape
    if D2 != D or tuple(out.shape) != tuple(q.shape) or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    dt = k_pool.dtype
    ws_ptr, ws_bytes = C.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    check(lib.pa_decode(_dev(out, "out", dt), _dev(q, "q", dt), _dev(k_pool, "k_pool", dt),
                        _dev(v_pool, "v_pool", dt), N, _dev(block_tables, "block_tables", torch.int32),
                        block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32), B, Hq, Hkv, D, b,
                        float(scale), int(partition_tokens), ws_ptr, ws_bytes, _dtype_id(k_pool),
                        _stream(stream)), "pa_decode")


def pa_prefill(out, q, k_pool, v_pool, block_tables, seq_lens, qstart, scale, max_query_len=None,
               stream=None) -> None:
    """Causal attention of each sequence's chunk (rows qstart[s] .. qstart[s+1]-1 of
    q [total_q, Hq, D]) over its paged history plus the chunk; seq_lens [B] are the
    total lengths (chunk included), qstart [B+1] int32.  ``max_query_len`` is the
    largest chunk (read from qstart, with a device sync, when None)."""
    lib = load()
    T, Hq, D = q.shape
    N, Hkv, b, D2 = k_pool.shape
    if D2 != D or tuple(out.shape) != tuple(q.shape) or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    B = seq_lens.shape[0]
    if block_tables.dim() != 2 or block_tables.shape[0] != B or qstart.shape != (B + 1,):
        raise ValueError("block_tables must be [B, max_blocks], seq_lens [B] and qstart [B + 1]")
    if max_query_len is None:
        max_query_len = int((qstart[1:] - qstart[:-1]).max().item()) if B else 0
    dt = k_pool.dtype
    check(lib.pa_prefill(_dev(out, "out", dt), _dev(q, "q", dt), _dev(k_pool, "k_pool", dt),
                         _dev(v_pool, "v_pool", dt), N, _dev(block_tables, "block_tables", torch.int32),
                         block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32),
                         _dev(qstart, "qstart", torch.int32), B, T, int(max_query_len), Hq, Hkv, D, b, float(scale),
                         _dtype_id(k_pool), _stream(stream)), "pa_prefill")


def pa_decode_append(out, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables, seq_lens, scale,
                     partition_tokens=0, workspace=None, stream=None) -> None:
    """pa_kv_append of each sequence's newest row (k_new, v_new [B, Hkv, D] at
    slot_mapping [B] int64, the slot of position seq_lens[s] - 1) followed by
    pa_decode; one launch for fp16 / bf16 pools on the tensor-core kernel."""
    lib = load()
    B, Hq, D = q.shape
    N, Hkv, b, D2 = k_pool.shape
    if D2 != D or tuple(out.shape) != tuple(q.shape) or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D) or slot_mapping.shape != (B,):
        raise ValueError("k_new, v_new must be [B, Hkv, D] and slot_mapping [B]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    dt = k_pool.dtype
    ws_ptr, ws_bytes = C.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    check(lib.pa_decode_append(_dev(out, "out", dt), _dev(q, "q", dt), _dev(k_new, "k_new", dt),
                               _dev(v_new, "v_new", dt), _dev(slot_mapping, "slot_mapping", torch.int64),
                               _dev(k_pool, "k_pool", dt), _dev(v_pool, "v_pool", dt), N,
                               _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                               _dev(seq_lens, "seq_lens", torch.int32), B, Hq, Hkv, D, b, float(scale),
                               int(partition_tokens), ws_ptr, ws_bytes, _dtype_id(k_pool), _stream(stream)),
          "pa_decode_append")


def pa_decode_noalloc(out, q, k_pool, v_pool, block_tables, seq_lens, scale, partition_tokens=0,
                      stream=None) -> None:
    """pa_decode with the library's fixed scratch array instead of caller scratch
    (for callers that cannot allocate device memory); raises PagedKVError
    (PA_ERR_INVALID) when the batch needs more scratch than the array holds."""
    lib = load()
    B, Hq, D = q.shape
    N, Hkv, b, D2 = k_pool.shape
    if D2 != D or tuple(out.shape) != tuple(q.shape) or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    dt = k_pool.dtype
    check(lib.pa_decode_noalloc(_dev(out, "out", dt), _dev(q, "q", dt), _dev(k_pool, "k_pool", dt),
                                _dev(v_pool, "v_pool", dt), N, _dev(block_tables, "block_tables", torch.int32),
                                block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32), B, Hq, Hkv, D, b,
                                float(scale), int(partition_tokens), _dtype_id(k_pool), _stream(stream)),
          "pa_decode_noalloc")


def pa_kv_append_fp8(k, v, k_pool, v_pool, k_scale, v_scale, slot_mapping, stream=None) -> None:
    """Quantise k, v [T, Hkv, D] (f32/f16/bf16) to E4M3 bytes of pools
    [N, Hkv, b, D] (uint8) with per-head scales k_scale, v_scale [Hkv] (f32)."""
    lib = load()
    N, Hkv, b, D = k_pool.shape
    if k_pool.dtype != torch.uint8 or v_pool.dtype != torch.uint8 or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("FP8 pools are uint8 tensors [N, Hkv, b, D]")
    if k.shape != v.shape or k.dim() != 3 or k.shape[1:] != (Hkv, D) or slot_mapping.shape != (k.shape[0],):
        raise ValueError("shape mismatch: k, v [T, Hkv, D]; slots [T]")
    if k_scale.shape != (Hkv,) or v_scale.shape != (Hkv,):
        raise ValueError("scales are [Hkv]")
    check(lib.pa_kv_append_fp8(_dev(k, "k", k.dtype), _dev(v, "v", k.dtype), _dtype_id(k), _dev(k_pool, "k_pool"),
                               _dev(v_pool, "v_pool"), _dev(k_scale, "k_scale", torch.float32),
                               _dev(v_scale, "v_scale", torch.float32),
                               _dev(slot_mapping, "slot_mapping", torch.int64), k.shape[0], N, Hkv, D, b,
                               _stream(stream)), "pa_kv_append_fp8")


def pa_decode_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, scale, partition_tokens=0,
                  workspace=None, stream=None) -> None:
    """Decode over E4M3 pools [N, Hkv, b, D] (uint8) with per-head scales;
    q, out [B, Hq, D] in f16 or bf16."""
    lib = load()
    B, Hq, D = q.shape
    N, Hkv, b, D2 = k_pool.shape
    if D2 != D or tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype:
        raise ValueError("shape mismatch between q, out and the pools")
    if k_pool.dtype != torch.uint8 or v_pool.dtype != torch.uint8 or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("FP8 pools are uint8 tensors [N, Hkv, b, D]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    ws_ptr, ws_bytes = C.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    check(lib.pa_decode_fp8(_dev(out, "out", q.dtype), _dev(q, "q", q.dtype), _dtype_id(q), _dev(k_pool, "k_pool"),
                            _dev(v_pool, "v_pool"), _dev(k_scale, "k_scale", torch.float32),
                            _dev(v_scale, "v_scale", torch.float32), N,
                            _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                            _dev(seq_lens, "seq_lens", torch.int32), B, Hq, Hkv, D, b, float(scale),
                            int(partition_tokens), ws_ptr, ws_bytes, _stream(stream)), "pa_decode_fp8")


DECODE_KERNELS = {"auto": 0, "simt": 1, "mma": 2}


def pa_set_decode_kernel(kernel: str) -> None:
    """Process-wide choice of the decode kernel: "auto", "simt" or "mma"."""
    check(load().pa_set_decode_kernel(DECODE_KERNELS[kernel]), "pa_set_decode_kernel")


def pa_set_decode_heads_per_cta(heads: int) -> None:
    """KV heads per CTA of the tensor-core decode kernel: 0 (choose per launch), 1 or 2."""
    check(load().pa_set_decode_heads_per_cta(int(heads)), "pa_set_decode_heads_per_cta")


def pa_get_device_error(stream=None) -> int:
    """Synchronise the stream, read and clear the device error word (PA_DEVERR_* bits)."""
    lib = load()
    code = C.c_int(0)
    st = lib.pa_get_device_error(C.byref(code), _stream(stream))
    if st not in (0, 4, 5):
        check(st, "pa_get_device_error")
    return code.value


def pa_status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()
