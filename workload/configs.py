"""Seeded synthetic workloads for paged decode (five configurations).

A workload is pure input data: shapes, the initial free-list order of the
block pool, and a list of host operations ("ops") that a driver applies to a
block manager.  Both the GPU path and the oracle replay the same ops with
their own block manager and their own kernels; this module computes no block
table, slot, copy pair or attention value itself.

Op vocabulary (tuples):
  ("create", uid)                 new empty sequence
  ("write", uid, n)               reserve n new positions, then append the K/V
                                  rows of positions [len, len + n)
  ("fork", parent_uid, child_uid) child aliases the parent's blocks
  ("truncate", uid, length)       roll back to ``length`` tokens
  ("free", uid)                   release every block of the sequence
  ("step", (uid, ...))            one decode step for this batch: reserve one
                                  position per sequence, copy-on-write copies,
                                  append one K/V row per sequence, then attend
                                  over the new length with one query each.

Token contents are addressed, not stored: the K (or V) row at position ``p``
of sequence ``uid`` in ``layer`` is ``kv_rows(wl, layer, kind, owner, p)``
where ``owner = wl.content_owner(uid, p)`` (a shared system prefix is owned by
the sequence that wrote it).  The query of batch row ``r`` at decode step
``s`` is ``q_rows(wl, layer, s, r)``.  Values are approximately N(0, 1)
(see ``workload.rng``) rounded once to the storage dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

from . import rng

_TAG_K, _TAG_V, _TAG_Q = 11, 12, 13
POS_BITS = 17  # positions < 131072
UID_LIMIT = 1 << 20

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    cid: int
    name: str
    Hq: int
    Hkv: int
    D: int
    b: int
    dtype: str
    num_blocks: int
    layers: int
    seed: int
    free_order: np.ndarray            # int32 permutation of range(num_blocks)
    setup_ops: list = field(default_factory=list)
    step_ops: list = field(default_factory=list)   # list (per decode step) of op lists
    partition_tokens: int = 0         # decode partition tokens (0: the library's automatic size)
    prefix_owner: int = -1            # uid owning shared prefix content (-1: none)
    prefix_len: int = 0
    tolerance: float = 0.0            # max-abs tolerance of attention vs fp64

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def elt(self) -> int:
        return torch.tensor([], dtype=self.torch_dtype).element_size()

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def content_owner(self, uid: int, pos: int) -> int:
        if self.prefix_owner >= 0 and pos < self.prefix_len:
            return self.prefix_owner
        return uid

    def content_owners(self, uid: int, positions: np.ndarray) -> np.ndarray:
        own = np.full(positions.shape, uid, dtype=np.int64)
        if self.prefix_owner >= 0:
            own[positions < self.prefix_len] = self.prefix_owner
        return own


# --------------------------------------------------------------------------- values

def kv_rows(wl: Workload, layer: int, kind: str, owners, positions, heads=None,
            device="cpu") -> torch.Tensor:
    """K (kind='k') or V (kind='v') rows [T, len(heads), D] in the storage dtype."""
    owners = torch.as_tensor(np.asarray(owners, dtype=np.int64), device=device)
    positions = torch.as_tensor(np.asarray(positions, dtype=np.int64), device=device)
    if heads is None:
        heads = torch.arange(wl.Hkv, device=device, dtype=torch.int64)
    else:
        heads = torch.as_tensor(np.asarray(heads, dtype=np.int64), device=device)
    key = rng.stream_key(wl.seed, _TAG_K if kind == "k" else _TAG_V, layer)
    d = torch.arange(wl.D, device=device, dtype=torch.int64)
    row = (owners << POS_BITS) + positions                      # [T]
    idx = ((row[:, None, None] * wl.Hkv + heads[None, :, None]) * wl.D + d[None, None, :])
    return rng.normal_from_index(key, idx).to(wl.torch_dtype)


def kv_scales(wl: Workload, layer: int, kind: str) -> np.ndarray:
    """fp32 [Hkv] scales of an FP8 (E4M3) K or V pool: 1/32, spread slightly by
    head and layer (values of about N(0, 1) then use codes up to ~110 of 448)."""
    h = np.arange(wl.Hkv, dtype=np.float64)
    base = 1.0 / 32 if kind == "k" else 1.0 / 30
    return (base * (1.0 + 0.05 * h + 0.01 * layer)).astype(np.float32)


def q_rows(wl: Workload, layer: int, step: int, rows, device="cpu") -> torch.Tensor:
    """Query rows [len(rows), Hq, D] for decode step ``step`` in the storage dtype."""
    rows = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=device)
    key = rng.stream_key(wl.seed, _TAG_Q, layer)
    h = torch.arange(wl.Hq, device=device, dtype=torch.int64)
    d = torch.arange(wl.D, device=device, dtype=torch.int64)
    base = (int(step) << 13) + rows                                # rows < 8192
    idx = ((base[:, None, None] * wl.Hq + h[None, :, None]) * wl.D + d[None, None, :])
    return rng.normal_from_index(key, idx).to(wl.torch_dtype)


# --------------------------------------------------------------------------- configs

def _perm(seed: int, n: int) -> np.ndarray:
    return np.random.default_rng(seed).permutation(n).astype(np.int32)


def config1() -> Workload:
    """Tiny correctness case (fp32): histories {1,7,16,33}, one decode step."""
    seed = 1001
    wl = Workload(1, "tiny-f32", Hq=4, Hkv=2, D=64, b=16, dtype="f32", num_blocks=16,
                  layers=1, seed=seed, free_order=_perm(seed, 16), tolerance=1e-5)
    for uid, L in enumerate([1, 7, 16, 33]):
        wl.setup_ops += [("create", uid), ("write", uid, L)]
    wl.step_ops = [[("step", (0, 1, 2, 3))]]
    return wl


def config2(steps: int = 64) -> Workload:
    """Llama-3-8B-shaped layer, bf16, 32 sequences of 20..500 tokens, 64 steps."""
    seed = 1002
    r = np.random.default_rng(seed)
    lens = r.integers(20, 501, size=32)
    wl = Workload(2, "llama8b-bf16-b32", Hq=32, Hkv=8, D=128, b=16, dtype="bf16",
                  num_blocks=4096, layers=1, seed=seed, free_order=_perm(seed + 7, 4096),
                  tolerance=1e-2)
    for uid, L in enumerate(lens):
        wl.setup_ops += [("create", uid), ("write", uid, int(L))]
    batch = tuple(range(32))
    wl.step_ops = [[("step", batch)] for _ in range(steps)]
    return wl


def config3(steps: int = 1, layers: int = 32, batch: int = 8, hist: int = 32767) -> Workload:
    """Long context, fp16: 8 x 32768 tokens, 32 layers, 20000-block pool per layer."""
    seed = 1003
    wl = Workload(3, "longctx-f16-b8x32k", Hq=32, Hkv=8, D=128, b=16, dtype="f16",
                  num_blocks=20000, layers=layers, seed=seed,
                  free_order=_perm(seed, 20000), tolerance=2e-3, partition_tokens=512)
    for uid in range(batch):
        wl.setup_ops += [("create", uid), ("write", uid, hist)]
    wl.step_ops = [[("step", tuple(range(batch)))] for _ in range(steps)]
    return wl


def config4(steps: int = 1, batch: int = 256, num_blocks: int = 65536) -> Workload:
    """Prefix-shared mixed batch, bf16: 256 sequences share a 512-token prefix.

    Lengths are log-uniform in [128, 8192], clamped to at least 513 so that every
    sequence holds the whole prefix plus one private token; sequence 0 is then
    truncated to 500 tokens, leaving the last prefix block shared and partially
    filled from its own view, so its next append triggers a copy-on-write.
    """
    seed = 1004
    r = np.random.default_rng(seed)
    lens = np.exp(r.uniform(math.log(128), math.log(8192), size=batch))
    lens = np.maximum(np.floor(lens).astype(np.int64), 513)
    wl = Workload(4, "prefix-shared-bf16-b256", Hq=32, Hkv=8, D=128, b=16, dtype="bf16",
                  num_blocks=num_blocks, layers=1, seed=seed,
                  free_order=_perm(seed, num_blocks), prefix_owner=0, prefix_len=512,
                  tolerance=1e-2)
    ops = [("create", 0), ("write", 0, 512)]
    for uid in range(1, batch):
        ops.append(("fork", 0, uid))
    for uid in range(batch):
        ops.append(("write", uid, int(lens[uid]) - 512))
    ops.append(("truncate", 0, 500))
    wl.setup_ops = ops
    wl.step_ops = [[("step", tuple(range(batch)))] for _ in range(steps)]
    return wl


CONFIG5_COMBOS = [(D, G, b, dt) for D in (64, 128, 256) for G in (1, 4, 8)
                  for b in (16, 32) for dt in ("f16", "bf16")]


def config5(D: int = 128, G: int = 4, b: int = 16, dtype: str = "bf16", steps: int = 200,
            batch: int = 128, p_finish: float = 0.01, prompt: int = 64) -> Workload:
    """Head-shape / block-size sweep with continuous batching (one combo).

    Each step every live sequence finishes with probability ``p_finish`` and
    releases its blocks; a replacement arrives in its batch row with a
    ``prompt``-token prompt, so the pool fragments.
    """
    combo = CONFIG5_COMBOS.index((D, G, b, dtype))
    seed = 1005 * 1000 + combo
    r = np.random.default_rng(seed)
    Hq = 32
    Hkv = Hq // G
    nb = 32768 if b == 16 else 16384
    tol = 2e-3 if dtype == "f16" else 1e-2
    wl = Workload(5, f"sweep-D{D}-G{G}-b{b}-{dtype}", Hq=Hq, Hkv=Hkv, D=D, b=b, dtype=dtype,
                  num_blocks=nb, layers=1, seed=seed, free_order=_perm(seed + 7, nb),
                  tolerance=tol)
    lens = r.integers(1, 4097, size=batch)
    for uid in range(batch):
        wl.setup_ops += [("create", uid), ("write", uid, int(lens[uid]))]
    live = list(range(batch))
    next_uid = batch
    for _s in range(steps):
        ops = []
        fin = r.random(batch) < p_finish
        for row in np.nonzero(fin)[0]:
            ops += [("free", live[row]), ("create", next_uid), ("write", next_uid, prompt)]
            live[row] = next_uid
            next_uid += 1
        ops.append(("step", tuple(live)))
        wl.step_ops.append(ops)
    return wl


def all_configs():
    return {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


# --------------------------------------------------------------------------- prefill

@dataclass
class PrefillWorkload:
    """Chunked prefill of a Llama-3-8B-shaped layer: every sequence holds
    ``history`` cached tokens and attends a ``chunk`` of new ones causally.
    Blocks are scattered over the pool by a seeded permutation; K, V and q are
    N(0, 1) rounded to the dtype (``prefill_inputs``)."""
    name: str
    Hq: int
    Hkv: int
    D: int
    b: int
    dtype: str
    batch: int
    history: int
    chunk: int
    num_blocks: int
    seed: int

    @property
    def length(self) -> int:
        return self.history + self.chunk

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def tables(self) -> np.ndarray:
        """int32 [batch, blocks per sequence] drawn from a seeded permutation of the pool."""
        per = -(-self.length // self.b)
        return _perm(self.seed, self.num_blocks)[:self.batch * per].reshape(self.batch, per)

    def qstart(self) -> np.ndarray:
        return (np.arange(self.batch + 1) * self.chunk).astype(np.int32)

    def causal_pairs(self) -> int:
        """(query row, visible key) pairs per query head: sum over the chunk of
        history + r + 1."""
        C, H = self.chunk, self.history
        return self.batch * (C * H + C * (C + 1) // 2)


def prefill_config(dtype: str = "bf16", batch: int = 8, history: int = 3072, chunk: int = 1024,
                   head_dim: int = 128) -> PrefillWorkload:
    """The Llama-3-8B layer shape (Hq 32, Hkv 8, D 128); other head dims keep the head counts."""
    per = -(-(history + chunk) // 16)
    shape = "llama8b" if head_dim == 128 else f"hq32-hkv8-d{head_dim}"
    return PrefillWorkload(f"prefill-{shape}-{dtype}-b{batch}-h{history}-c{chunk}", Hq=32, Hkv=8, D=head_dim, b=16,
                           dtype=dtype, batch=batch, history=history, chunk=chunk,
                           num_blocks=max(4096, batch * per + 64), seed=1006)


def prefill_inputs(wl: PrefillWorkload, device="cpu"):
    """Pools [N, Hkv, b, D] and packed q [batch * chunk, Hq, D] (seeded N(0, 1))."""
    g = torch.Generator(device=device).manual_seed(wl.seed)
    shape = (wl.num_blocks, wl.Hkv, wl.b, wl.D)
    k = torch.randn(shape, generator=g, device=device).to(wl.torch_dtype)
    v = torch.randn(shape, generator=g, device=device).to(wl.torch_dtype)
    q = torch.randn((wl.batch * wl.chunk, wl.Hq, wl.D), generator=g, device=device).to(wl.torch_dtype)
    return k, v, q
