"""Paged prefill in fp64 (test infrastructure, like the rest of ``oracle/``).

A chunk of new query tokens of one sequence attends causally to that
sequence's paged history plus the chunk itself ([P1] "Stretch exercises",
item 4, names the operation).  [P5] "4.1 How PagedAttention Reads KV", step 3,
gives the causal form: the query at global position i scores every key at
position p through the block table, keys with p > i get -inf, and

    o_i = sum_{p <= i} softmax_p(scale * q_i . k_p) v_p

which is decode attention over the first i + 1 positions.  The oracle is that
definition, one query row at a time, on the history gathered through the
table (``attention.gather_history``).

Readings (the pages leave these open):
  * chunked prefill: the chunk holds the LAST C positions of a sequence of
    total length L, whose K/V rows are already in the pool; chunk row r is at
    global position L - C + r and sees positions 0 .. L - C + r;
  * query head h reads KV head h // G, and the scale is the caller's, as for
    decode;
  * a batch packs its queries: sequence s owns rows qstart[s] .. qstart[s+1]
    of q (qstart holds B + 1 cumulative row counts).
"""
from __future__ import annotations

import numpy as np

from .attention import decode_attention, gather_history


def prefill_attention(q, K, V, scale: float) -> np.ndarray:
    """Causal attention of the C chunk rows q [C, Hq, D] over a contiguous
    history K, V [L, Hkv, D] whose last C rows are the chunk's own."""
    q = np.asarray(q, dtype=np.float64)
    C = q.shape[0]
    L = K.shape[0]
    if C > L:
        raise ValueError("the chunk is longer than the sequence")
    out = np.zeros(q.shape, dtype=np.float64)
    for r in range(C):
        visible = L - C + r + 1
        out[r] = decode_attention(q[r], K[:visible], V[:visible], scale)
    return out


def paged_prefill(q, k_pool, v_pool, table, length: int, block_size: int, scale: float) -> np.ndarray:
    """One sequence: gather its ``length`` positions through the table, then
    the causal definition for the chunk rows q [C, Hq, D]."""
    K = gather_history(k_pool, table, length, block_size)
    V = gather_history(v_pool, table, length, block_size)
    return prefill_attention(q, K, V, scale)


def paged_prefill_batch(q, k_pool, v_pool, tables, lengths, qstart, block_size: int, scale: float) -> np.ndarray:
    """Packed batch: rows qstart[s] .. qstart[s+1] of q [T, Hq, D] are the
    chunk of sequence s (total length lengths[s], table tables[s])."""
    q = np.asarray(q, dtype=np.float64)
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(len(lengths)):
        a, b = int(qstart[s]), int(qstart[s + 1])
        if b > a:
            out[a:b] = paged_prefill(q[a:b], k_pool, v_pool, tables[s], int(lengths[s]), block_size, scale)
    return out
