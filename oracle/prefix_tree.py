"""Prefix tree of cached full blocks: the radix-tree form of the prefix cache.

TEST INFRASTRUCTURE (oracle).  Sources: [P1] "25. Paged attention and
prefix caching", "Prefix caching" (closing paragraph: RadixAttention
generalises the prefix table to a radix tree over all cached prefixes);
[P2] "Модуль 09", "RadixAttention: более агрессивный кузен PagedAttention"
(the shared prefixes of all past requests form a tree that is searched
automatically and kept by least-recently-used eviction, outliving the
requests).  The pages give no algorithm; the readings taken:

  * one node per full block of b tokens, the edge into it labelled by the
    block's b token ids; the root is the empty prefix.  A node therefore
    stands for the whole prefix on the path to it (the flat table's key),
    and a radix tree's merging of single-child chains would change no
    decision, so nodes stay one block each;
  * attach: from the root, follow the child labelled by the prompt's next
    full block while one exists, leaving at least one prompt token to
    prefill (the flat table's rule); each matched node's block gains the new
    sequence as a holder, and each matched node becomes the most recently
    used, in walk order;
  * remember: walk the sequence's full blocks; descend through a child that
    exists (without touching it, as the flat table leaves an existing
    entry's position alone), otherwise hang a new child holding the
    sequence's block there (the tree takes its own reference; the node is
    most recently used);
  * evict: only leaves go -- a node whose prefix no cached child extends --
    least recently used first, and only while the tree alone holds the
    block; a parent whose last child went becomes a leaf and a candidate in
    turn.  This is where the tree differs from the flat table, which may
    drop an inner prefix and strand the longer ones behind it.

Invariants (checked by the pins): every node's parent is in the tree
(prefix-closed), every cached block has a holder count of at least one,
counts equal holders (tables plus tree nodes), free + live = N.
"""
from __future__ import annotations

from .blocks import SeqTables


class _Node:
    __slots__ = ("parent", "label", "block", "children", "used")

    def __init__(self, parent, label, block, used):
        self.parent = parent
        self.label = label          # tuple of the block's b token ids (None at the root)
        self.block = block          # physical block id (-1 at the root)
        self.children = {}          # label -> _Node
        self.used = used            # recency stamp: larger = more recently used


class BlockPrefixTree:
    """Cached full blocks as a tree of block-labelled edges over one SeqTables."""

    def __init__(self, tables: SeqTables):
        self.tables = tables
        self.root = _Node(None, None, -1, 0)
        self.clock = 0

    def _stamp(self) -> int:
        self.clock += 1
        return self.clock

    def _labels(self, tokens):
        b = self.tables.block_size
        return [tuple(tokens[i:i + b]) for i in range(0, len(tokens) - b + 1, b)]

    def nodes(self):
        """Every cached node (root excluded), parents before children."""
        out, stack = [], list(self.root.children.values())
        while stack:
            n = stack.pop()
            out.append(n)
            stack.extend(n.children.values())
        return out

    def cached_blocks(self) -> list:
        return sorted(n.block for n in self.nodes())

    def attach(self, seq, prompt) -> int:
        """Create ``seq`` holding the cached blocks along the prompt's path; returns the
        tokens reused (a multiple of b, at most len(prompt) - 1)."""
        prompt = list(prompt)
        b = self.tables.block_size
        usable = max(0, (len(prompt) - 1) // b)
        path, node = [], self.root
        for label in self._labels(prompt)[:usable]:
            child = node.children.get(label)
            if child is None:
                break
            path.append(child)
            node = child
        self.tables.create(seq)
        for n in path:
            n.used = self._stamp()
            self.tables.allocator.share(n.block)
        self.tables.tables[seq] = [n.block for n in path]
        self.tables.lengths[seq] = len(path) * b
        return len(path) * b

    def remember(self, seq, tokens) -> None:
        """Hang the full blocks of ``seq`` (holding ``tokens``) below their cached prefix."""
        table = self.tables.tables[seq]
        node = self.root
        for i, label in enumerate(self._labels(list(tokens))):
            child = node.children.get(label)
            if child is None:
                self.tables.allocator.share(table[i])
                child = _Node(node, label, table[i], self._stamp())
                node.children[label] = child
            node = child

    def evict(self, blocks_wanted: int) -> None:
        """Drop least-recently-used leaves held only by the tree until ``blocks_wanted``
        blocks are free or no such leaf is left."""
        alloc = self.tables.allocator
        while alloc.num_free < int(blocks_wanted):
            idle = [n for n in self.nodes() if not n.children and alloc.refs[n.block] == 1]
            if not idle:
                return
            victim = min(idle, key=lambda n: n.used)
            del victim.parent.children[victim.label]
            alloc.release(victim.block)
