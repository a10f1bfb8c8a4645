"""Oracle for paged decode: a plain, slow, obviously correct CPU restatement.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code with the CUDA path (``paged_kv_cache_66_gb300``); the two
meet only in the seeded input generator ``workload``.

Sources restated here (cited by page title and section):
  [P1] "25. Paged attention and prefix caching" (inference.shantanugoel.com)
  [P2] "Модуль 09: PagedAttention: пейджинг KV-кэша" (hermes-agent.ru)
  [P4] "PagedAttention and the KV Cache" (kanthi.in)
  [P5] "Chapter 7 Paged KV Cache and Memory Management" (zero-to-sglang)

Modules:
  blocks     -- BlockAllocator, SeqTables, KeyedPrefixIndex / PrefixTable
                ([P1] allocator, paged cache, prefix caching; written from the
                invariants the pages fix, readings in the module header)
  prefix_hash -- SHA-256 chain keys and the prefix table keyed by them ([P1] prefix caching)
  prefix_tree -- the block prefix tree, the radix-tree form of the prefix cache
  cache_ops  -- K/V scatter through slots and block copy-on-write ([P1] update/reserve)
  attention  -- decode attention by its definition (fp64), the blockwise
                online-softmax / split merge used only as a cross-check ([P5] 4.2)
  driver     -- replays a ``workload`` op list through the above

Every function here is pinned by ``tests/test_oracle_pins.py`` to values the
pages print, closed forms, brute force or library routines.
"""
from . import attention, blocks, cache_ops, driver  # noqa: F401
