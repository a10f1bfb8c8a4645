"""Decode attention over a paged history, in fp64.

The oracle is the plain definition: gather the sequence's K/V history through
its block table into a contiguous array, then

    s_t   = scale * sum_d q[h, d] * K[t, h // G, d]        t = 0 .. L-1
    p_t   = exp(s_t - max_t s_t)
    out_h = sum_t p_t * V[t, h // G, :] / sum_t p_t

([P2] "5. Внимание по страницам" and its reference_attention; [P4] "KV cache
in Transformers (reminder)"; [P1] "Attention that reads through the table":
query head h reads KV head h // group, scale = 1 / sqrt(d) supplied by the
caller).  [P5] "4.2 Proof of Mathematical Equivalence" shows that the
blockwise online-softmax method reaches exactly this value, so the definition
is the oracle.  Inputs are the stored (already rounded) q, K, V values,
promoted to fp64.

The blockwise online-softmax with a split-K partition merge is restated here
too (``decode_attention_split``), only as a cross-check of the merge algebra of
[P5] 4.2 ("Block Merging Mechanism of Online Softmax").

Reading: a sequence of length 0 (outside the pages' precondition L >= 1)
yields a zero output row.
"""
from __future__ import annotations

import numpy as np


def gather_history(pool, table, length: int, block_size: int) -> np.ndarray:
    """Contiguous [L, Hkv, D] fp64 history: row t = pool[table[t // b], :, t % b, :].

    [P2] "Код" (gather_kv); [P5] "3.2 How Logical Blocks Map to Physical Blocks",
    step 3.
    """
    pool = np.asarray(pool.float().numpy() if hasattr(pool, "float") else pool)
    t = np.arange(length)
    blocks = np.asarray(table, dtype=np.int64)[t // block_size]
    return pool[blocks, :, t % block_size, :].astype(np.float64)    # [L, Hkv, D]


def decode_attention(q, K, V, scale: float) -> np.ndarray:
    """Attention of one query per head over a contiguous history (definition).

    q [Hq, D]; K, V [L, Hkv, D]; returns [Hq, D] fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, D = q.shape
    L, Hkv, _ = K.shape
    group = Hq // Hkv
    out = np.zeros((Hq, D), dtype=np.float64)
    if L == 0:
        return out
    for h in range(Hq):
        g = h // group
        s = scale * (K[:, g, :] @ q[h])
        p = np.exp(s - s.max())
        out[h] = (p @ V[:, g, :]) / p.sum()
    return out


def paged_decode(q, k_pool, v_pool, table, length: int, block_size: int, scale: float):
    """Paged decode for one sequence: gather through the table, then the definition."""
    K = gather_history(k_pool, table, length, block_size)
    V = gather_history(v_pool, table, length, block_size)
    return decode_attention(q, K, V, scale)


# ----------------------------------------------------------------- cross-check only

def local_statistics(s, Vb):
    """Block-local (m, l, O) of one query over the valid tokens of one block.

    [P5] 4.2: m_j = max_t s_t, l_j = sum_t exp(s_t - m_j), O_j = sum_t exp(s_t - m_j) v_t.
    """
    m = s.max()
    w = np.exp(s - m)
    return m, w.sum(), w @ Vb


def merge(a, b):
    """Merge two (m, l, O) states onto the new reference max ([P5] 4.2, steps 1-3).

    A state with l == 0 (fully masked: m = -inf) contributes nothing.
    """
    (ma, la, Oa), (mb, lb, Ob) = a, b
    if la == 0:
        return b
    if lb == 0:
        return a
    m = max(ma, mb)
    fa, fb = np.exp(ma - m), np.exp(mb - m)
    return m, la * fa + lb * fb, Oa * fa + Ob * fb


def decode_attention_split(q, K, V, scale: float, block_size: int, partition_tokens: int):
    """Online softmax block by block inside each partition, then a merge of the
    partitions (flash-decoding split), in fp64.  A partition or block with no
    valid token contributes nothing and is left out of the merge ([P5] 4.2)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, D = q.shape
    L, Hkv, _ = K.shape
    group = Hq // Hkv
    out = np.zeros((Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        total = (-np.inf, 0.0, np.zeros(D))
        for p0 in range(0, L, partition_tokens):
            part = (-np.inf, 0.0, np.zeros(D))
            for b0 in range(p0, min(L, p0 + partition_tokens), block_size):
                b1 = min(L, b0 + block_size)
                s = scale * (K[b0:b1, g, :] @ q[h])
                part = merge(part, local_statistics(s, V[b0:b1, g, :]))
            total = merge(total, part)
        m, l, O = total
        if l > 0:
            out[h] = O / l
    return out
