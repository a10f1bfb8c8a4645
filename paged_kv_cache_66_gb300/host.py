"""Python binding of the host block manager (include/pagedkv_host.h).

Status codes become the exceptions the pages use for the same events
("25. Paged attention and prefix caching"): pool exhaustion -> MemoryError,
over-release -> RuntimeError, duplicate sequence -> ValueError; an unknown
sequence id -> KeyError.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from ._lib import PagedKVError, load

_P64 = C.POINTER(C.c_int64)
_P32 = C.POINTER(C.c_int32)


def _raise(st: int, what: str):
    if st == 0:
        return
    if st == 6:
        raise MemoryError(f"{what}: KV block pool exhausted")
    if st == 7:
        raise RuntimeError(f"{what}: block released more times than it was referenced")
    if st == 8:
        raise ValueError(f"{what}: sequence already exists")
    if st == 9:
        raise KeyError(f"{what}: unknown sequence")
    raise PagedKVError(st, what)


def _p64(a: np.ndarray):
    return a.ctypes.data_as(_P64)


def _p32(a: np.ndarray):
    return a.ctypes.data_as(_P32)


def prefix_salt(model_revision: str = "", adapter: str = "", extra=()) -> bytes:
    """Salt bytes for the hash-chain prefix table: every field that changes a
    block's K/V besides its tokens (model revision, adapter, multimodal input
    digests), each length-prefixed so that no two field lists share bytes."""
    out = bytearray()
    for field in (model_revision, adapter, *extra):
        b = field.encode() if isinstance(field, str) else bytes(field)
        out += len(b).to_bytes(8, "little") + b
    return bytes(out)


def prefix_chain_keys(tokens, block_size: int, salt: bytes = b"") -> list:
    """Hash-chain keys (32 bytes each) of the full blocks of ``tokens``."""
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    full = t.shape[0] // int(block_size) if int(block_size) > 0 else 0   # the library rejects block_size <= 0
    out = np.zeros(max(full, 1) * 32, dtype=np.uint8)
    salt = bytes(salt)
    _raise(load().pa_prefix_chain_keys(_p64(t), t.shape[0], int(block_size), salt, len(salt),
                                       out.ctypes.data_as(C.c_void_p)), "chain keys")
    return [out[32 * i:32 * (i + 1)].tobytes() for i in range(full)]


class HostBlockManager:
    """Free list + refcounts, per-sequence block tables, prefix table (C++)."""

    def __init__(self, num_blocks: int, block_size: int, initial_order=None):
        self._lib = load()
        order = None
        if initial_order is not None:
            self._order = np.ascontiguousarray(np.asarray(initial_order, dtype=np.int32))
            order = _p32(self._order)
        h = self._lib.pa_host_create(int(num_blocks), int(block_size), order)
        if not h:
            raise ValueError("invalid pool size, block size or initial order")
        self._h = C.c_void_p(h)
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self._pairs = np.zeros((64, 2), dtype=np.int64)
        self._n = np.zeros(1, dtype=np.int64)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pa_host_destroy(h)
            self._h = None

    # ------------------------------------------------------------ sequences
    def create(self, seq: int) -> None:
        _raise(self._lib.pa_host_seq_create(self._h, int(seq)), "create")

    def reserve(self, seq: int, new_tokens: int):
        cap = int(new_tokens) // self.block_size + 2
        if self._pairs.shape[0] < cap:
            self._pairs = np.zeros((cap, 2), dtype=np.int64)
        _raise(self._lib.pa_host_reserve(self._h, int(seq), int(new_tokens), _p64(self._pairs),
                                         self._pairs.shape[0], _p64(self._n)), "reserve")
        return [tuple(int(x) for x in r) for r in self._pairs[: int(self._n[0])]]

    def slots(self, seq: int, start: int, n: int) -> np.ndarray:
        out = np.zeros(int(n), dtype=np.int64)
        _raise(self._lib.pa_host_slots(self._h, int(seq), int(start), int(n), _p64(out)), "slots")
        return out

    def advance(self, seq: int, n: int) -> None:
        _raise(self._lib.pa_host_advance(self._h, int(seq), int(n)), "advance")

    def fork(self, parent: int, child: int) -> None:
        _raise(self._lib.pa_host_fork(self._h, int(parent), int(child)), "fork")

    def free(self, seq: int) -> None:
        _raise(self._lib.pa_host_free(self._h, int(seq)), "free")

    def truncate(self, seq: int, length: int) -> None:
        _raise(self._lib.pa_host_truncate(self._h, int(seq), int(length)), "truncate")

    def length(self, seq: int) -> int:
        out = np.zeros(1, dtype=np.int64)
        _raise(self._lib.pa_host_length(self._h, int(seq), _p64(out)), "length")
        return int(out[0])

    def table(self, seq: int) -> list:
        n = np.zeros(1, dtype=np.int64)
        st = self._lib.pa_host_table(self._h, int(seq), None, 0, _p64(n))
        if st not in (0, 1):
            _raise(st, "table")
        out = np.zeros(max(int(n[0]), 1), dtype=np.int32)
        _raise(self._lib.pa_host_table(self._h, int(seq), _p32(out), out.shape[0], _p64(n)), "table")
        return out[: int(n[0])].tolist()

    @property
    def num_free(self) -> int:
        return int(self._lib.pa_host_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.pa_host_refcount(self._h, int(block)))

    def batch(self, seqs, stride: int | None = None):
        seqs = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        B = seqs.shape[0]
        w = np.zeros(1, dtype=np.int64)
        if stride is None:
            st = self._lib.pa_host_batch(self._h, _p64(seqs), B, _p32(np.zeros(1, np.int32)), 0,
                                         _p32(np.zeros(max(B, 1), np.int32)), _p64(w))
            if st not in (0, 1):
                _raise(st, "batch")
            stride = int(w[0])
        tables = np.zeros((B, stride), dtype=np.int32)
        lens = np.zeros(B, dtype=np.int32)
        _raise(self._lib.pa_host_batch(self._h, _p64(seqs), B, _p32(tables), stride, _p32(lens), _p64(w)),
               "batch")
        return tables, lens

    def decode_step(self, seqs, tables_out: np.ndarray, lens_out: np.ndarray, slots_out: np.ndarray):
        """Reserve + slot + advance for one decode step, writing the padded tables
        (tables_out [B, stride] int32), lengths and slots in place.  Returns
        (copy pairs [n, 2] int64, width of the longest table)."""
        seqs = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        B = seqs.shape[0]
        if self._pairs.shape[0] < B + 1:
            self._pairs = np.zeros((B + 1, 2), dtype=np.int64)
        w = np.zeros(1, dtype=np.int64)
        _raise(self._lib.pa_host_decode_step(self._h, _p64(seqs), B, _p64(slots_out), _p64(self._pairs),
                                             self._pairs.shape[0], _p64(self._n), _p32(tables_out),
                                             tables_out.shape[1], _p32(lens_out), _p64(w)), "decode_step")
        return self._pairs[: int(self._n[0])].copy(), int(w[0])

    # ------------------------------------------------------------ prefix table
    def prefix_attach(self, seq: int, prompt) -> int:
        p = np.ascontiguousarray(np.asarray(prompt, dtype=np.int64))
        out = np.zeros(1, dtype=np.int64)
        _raise(self._lib.pa_host_prefix_attach(self._h, int(seq), _p64(p), p.shape[0], _p64(out)), "attach")
        return int(out[0])

    def prefix_remember(self, seq: int, tokens) -> None:
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        _raise(self._lib.pa_host_prefix_remember(self._h, int(seq), _p64(t), t.shape[0]), "remember")

    def prefix_evict(self, blocks_wanted: int) -> None:
        _raise(self._lib.pa_host_prefix_evict(self._h, int(blocks_wanted)), "evict")

    @property
    def prefix_entries(self) -> int:
        return int(self._lib.pa_host_prefix_entries(self._h))

    # ------------------------------------------------ hash-chain prefix table
    def hprefix_attach(self, seq: int, prompt, salt: bytes = b"") -> int:
        p = np.ascontiguousarray(np.asarray(prompt, dtype=np.int64))
        out = np.zeros(1, dtype=np.int64)
        salt = bytes(salt)
        _raise(self._lib.pa_host_hprefix_attach(self._h, int(seq), _p64(p), p.shape[0], salt, len(salt), _p64(out)),
               "attach")
        return int(out[0])

    def hprefix_remember(self, seq: int, tokens, salt: bytes = b"") -> None:
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        salt = bytes(salt)
        _raise(self._lib.pa_host_hprefix_remember(self._h, int(seq), _p64(t), t.shape[0], salt, len(salt)),
               "remember")

    def hprefix_evict(self, blocks_wanted: int) -> None:
        _raise(self._lib.pa_host_hprefix_evict(self._h, int(blocks_wanted)), "evict")

    @property
    def hprefix_entries(self) -> int:
        return int(self._lib.pa_host_hprefix_entries(self._h))

    def hprefix_blocks(self) -> list:
        """Cached block ids, least recently used first."""
        n = int(self._lib.pa_host_hprefix_blocks(self._h, None, 0))
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._lib.pa_host_hprefix_blocks(self._h, _p32(out), n)
        return out[:n].tolist()

    # ------------------------------------------------------ block prefix tree
    def tprefix_attach(self, seq: int, prompt) -> int:
        p = np.ascontiguousarray(np.asarray(prompt, dtype=np.int64))
        out = np.zeros(1, dtype=np.int64)
        _raise(self._lib.pa_host_tprefix_attach(self._h, int(seq), _p64(p), p.shape[0], _p64(out)), "attach")
        return int(out[0])

    def tprefix_remember(self, seq: int, tokens) -> None:
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        _raise(self._lib.pa_host_tprefix_remember(self._h, int(seq), _p64(t), t.shape[0]), "remember")

    def tprefix_evict(self, blocks_wanted: int) -> None:
        _raise(self._lib.pa_host_tprefix_evict(self._h, int(blocks_wanted)), "evict")

    @property
    def tprefix_nodes(self) -> int:
        return int(self._lib.pa_host_tprefix_nodes(self._h))

    def tprefix_blocks(self) -> list:
        """Cached block ids, ascending."""
        n = int(self._lib.pa_host_tprefix_blocks(self._h, None, 0))
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._lib.pa_host_tprefix_blocks(self._h, _p32(out), n)
        return out[:n].tolist()
