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
  * the table built on these keys (HashPrefixTable) is the generic prefix
    index of ``blocks`` with this key function: its attach / remember / evict
    rules are those of the tuple-keyed PrefixTable, so the two agree step for
    step whenever no two distinct prefixes share a key.
"""
from __future__ import annotations

import hashlib
import struct

from .blocks import KeyedPrefixIndex

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


class HashPrefixTable(KeyedPrefixIndex):
    """The prefix index of ``blocks`` with chain keys in place of token tuples.

    Every rule (which blocks attach may reuse, what remember publishes, which
    entries evict may drop, the LRU order) is the generic index's; only the
    key differs, so the two tables make the same decisions whenever no two
    distinct (salt, prefix) pairs share a key.
    """

    def block_keys(self, tokens, salt):
        key = root_key(salt)
        b = self.tables.block_size
        for start in range(0, len(tokens) - b + 1, b):
            key = next_key(key, tokens[start:start + b])
            yield key
