"""Hash-chain keys for automatic prefix caching (test infrastructure).

[P1] "Prefix caching": a cached block's key is the whole token prefix up to
the end of that block, because a block's K/V depend on every earlier token;
production engines hash the chain of block contents instead of keeping the
tuples, and the key must also cover whatever else changes the activations
(model revision, adapter, multimodal inputs).  [P2] "4. Prefix sharing и copy-on-write" says
the same of vLLM's automatic prefix caching (a block hashed by its tokens
and the hashes of the blocks before it); [P4] "Prefix sharing
(copy-on-write intuition)" likewise (block contents plus prefix identity).

Readings (the pages fix no hash function or byte layout):
  * the hash is SHA-256;
  * the chain starts from a root key that covers a caller-given salt (the
    bytes that identify model revision, adapter and multimodal inputs):
        root  = SHA-256(b"pagedkv.prefix.v1" || u64le(len(salt)) || salt)
  * full block i (tokens t[i*b : (i+1)*b]) has the key
        key_i = SHA-256(key_{i-1} || u32le(b) || i64le(t) for each token)
    with key_{-1} = root; a partial last block has no key;
  * the table built on these keys (HashPrefixTable) has exactly the attach /
    remember / evict rules of the tuple-keyed PrefixTable, so the two agree
    step for step whenever no two distinct prefixes share a key.
"""
from __future__ import annotations

import hashlib
import struct
from collections import OrderedDict

from .blocks import SeqTables

DOMAIN = b"pagedkv.prefix.v1"


def root_key(salt: bytes = b"") -> bytes:
    salt = bytes(salt)
    return hashlib.sha256(DOMAIN + struct.pack("<Q", len(salt)) + salt).digest()


def next_key(parent: bytes, block_tokens) -> bytes:
    block_tokens = [int(x) for x in block_tokens]
    payload = parent + struct.pack("<I", len(block_tokens)) + struct.pack(f"<{len(block_tokens)}q", *block_tokens)
    return hashlib.sha256(payload).digest()


def chain_keys(tokens, block_size: int, salt: bytes = b"") -> list:
    """Keys (32 bytes each) of the full blocks of ``tokens``."""
    tokens = list(tokens)
    keys, parent = [], root_key(salt)
    for i in range(len(tokens) // block_size):
        parent = next_key(parent, tokens[i * block_size:(i + 1) * block_size])
        keys.append(parent)
    return keys


class HashPrefixTable:
    """[P1]'s prefix cache with chain keys in place of token tuples.

    attach walks the prompt one full block at a time while the block's chain
    key is cached, sharing those blocks, and always leaves at least one
    prompt token to prefill; remember publishes the full blocks of a
    sequence (the cache takes its own reference); evict drops least-recently
    used entries whose block nobody else holds until enough blocks are free.
    """

    def __init__(self, tables: SeqTables):
        self.tables = tables
        self.entries: OrderedDict = OrderedDict()

    def attach(self, seq, prompt, salt: bytes = b"") -> int:
        t = self.tables
        t.create(seq)
        size, reused = t.block_size, 0
        prompt = list(prompt)
        key = root_key(salt)
        while reused + size <= len(prompt) - 1:
            key = next_key(key, prompt[reused:reused + size])
            block = self.entries.get(key)
            if block is None:
                break
            self.entries.move_to_end(key)
            t.allocator.share(block)
            t.tables[seq].append(block)
            reused += size
        t.lengths[seq] = reused
        return reused

    def remember(self, seq, tokens, salt: bytes = b"") -> None:
        t = self.tables
        for index, key in enumerate(chain_keys(tokens, t.block_size, salt)):
            if key not in self.entries:
                block = t.tables[seq][index]
                t.allocator.share(block)
                self.entries[key] = block

    def evict(self, blocks_wanted: int) -> None:
        t = self.tables
        for key in list(self.entries):
            if t.allocator.num_free >= blocks_wanted:
                break
            block = self.entries[key]
            if t.allocator.refs[block] == 1:
                del self.entries[key]
                t.allocator.release(block)
