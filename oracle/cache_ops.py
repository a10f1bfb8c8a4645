"""K/V pool writes: append through slots, and block copy-on-write.

Pools are plain torch CPU tensors in the storage dtype, laid out
[num_blocks, kv_heads, b, head_dim] per layer ([P1] "Paging": "per layer,
tensors of shape [num_blocks, kv_heads, b, head_dim]").  Element copies only,
so the results are exact.
"""
from __future__ import annotations

import torch


def new_pool(num_blocks: int, Hkv: int, b: int, D: int, dtype) -> torch.Tensor:
    """Zero-initialised pool; blocks are never zeroed again on allocation."""
    return torch.zeros((num_blocks, Hkv, b, D), dtype=dtype)


def append(k_pool: torch.Tensor, v_pool: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
           slots, block_size: int) -> None:
    """Write row t of ``k``/``v`` ([T, Hkv, D]) to (slot // b, :, slot % b, :).

    [P1] "The paged cache", update: new keys and values go to
    (table[p // b], :, p % b); here the caller has already resolved each
    position to its slot = block * b + offset.  Negative slots are skipped.
    """
    slots = torch.as_tensor(slots, dtype=torch.int64).reshape(-1)
    keep = slots >= 0
    block, off = slots[keep] // block_size, slots[keep] % block_size
    k_pool[block, :, off, :] = k[keep]
    v_pool[block, :, off, :] = v[keep]


def copy_blocks(k_pools, v_pools, pairs) -> None:
    """For each (src, dst): pool[dst] = pool[src] in every layer's K and V pool.

    [P1] "The paged cache", reserve: a shared block about to be written is
    copied into the fresh block in all layers' pools before the table is
    repointed.
    """
    for src, dst in pairs:
        for pool in list(k_pools) + list(v_pools):
            pool[int(dst)].copy_(pool[int(src)])
