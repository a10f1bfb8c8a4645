"""Host bookkeeping of the paged KV cache, restated from the pages.

[P1] "25. Paged attention and prefix caching", sections "Paging", "The
allocator", "The paged cache", "Sharing blocks: forks and copy-on-write",
"Prefix caching".

Readings where the pages differ or are silent:
  * free-list order: first-in first-out, as in [P1] "The allocator" (a deque
    popped at the front, released blocks appended at the back), seeded with a
    caller-given initial order.  ([P2] "Код" pops the end of a list instead.)
  * over-release: checked before the decrement; raises RuntimeError and leaves
    the state unchanged ([P2] "Код" asserts before decrementing; [P1] would
    leave the count at -1).
  * sharing a block that is not live (refcount 0) raises RuntimeError.
  * allocation failure inside ``reserve`` is all-or-nothing: the number of
    fresh blocks is counted first and MemoryError is raised before any state
    changes ([P1] raises from inside the loop).
  * no zeroing of a block on allocation ([P2] zeroes; [P1] does not).
"""
from __future__ import annotations

from collections import OrderedDict, deque


class BlockAllocator:
    """Free list plus per-block reference counts ([P1] "The allocator")."""

    def __init__(self, num_blocks: int, order=None):
        self.num_blocks = int(num_blocks)
        start = range(self.num_blocks) if order is None else [int(x) for x in order]
        if sorted(start) != list(range(self.num_blocks)):
            raise ValueError("initial order must be a permutation of the pool")
        self.free = deque(start)
        self.refs = [0] * self.num_blocks

    def allocate(self) -> int:
        if not self.free:
            raise MemoryError("KV block pool exhausted")
        block = self.free.popleft()
        self.refs[block] = 1
        return block

    def share(self, block: int) -> None:
        if self.refs[block] <= 0:
            raise RuntimeError(f"block {block} is not live")
        self.refs[block] += 1

    def release(self, block: int) -> None:
        if self.refs[block] <= 0:
            raise RuntimeError(f"block {block} released more times than it was referenced")
        self.refs[block] -= 1
        if self.refs[block] == 0:
            self.free.append(block)

    @property
    def num_free(self) -> int:
        return len(self.free)


class SeqTables:
    """Per-sequence block tables and lengths over one allocator.

    [P1] "The paged cache" (create, blocks_needed, reserve, set_batch, fork,
    free, truncate) without the tensors: copy-on-write returns the (source,
    destination) block pairs that the device must copy in every layer.
    """

    def __init__(self, num_blocks: int, block_size: int, order=None):
        self.allocator = BlockAllocator(num_blocks, order)
        self.block_size = int(block_size)
        self.tables: dict = {}
        self.lengths: dict = {}

    # [P1] "Paging": a sequence of L tokens needs ceil(L / b) blocks.
    def blocks_needed(self, tokens: int) -> int:
        return -(-int(tokens) // self.block_size)

    def create(self, seq) -> None:
        if seq in self.tables:
            raise ValueError(f"sequence {seq} already exists")
        self.tables[seq] = []
        self.lengths[seq] = 0

    def reserve(self, seq, new_tokens: int) -> list:
        """Make blocks exist for positions [length, length + new_tokens).

        A table entry in the written range whose block is shared (refcount > 1)
        is replaced by a fresh block: allocate, record the copy, release the old
        block, repoint ([P1] "The paged cache", reserve; "Sharing blocks").
        """
        table, start = self.tables[seq], self.lengths[seq]
        end = start + int(new_tokens)
        need = self.blocks_needed(end)
        first = start // self.block_size
        cow = [i for i in range(first, min(len(table), need))
               if self.allocator.refs[table[i]] > 1]
        grow = max(0, need - len(table))
        if len(cow) + grow > self.allocator.num_free:
            raise MemoryError("KV block pool exhausted")
        pairs = []
        for i in range(first, min(len(table), need)):
            old = table[i]
            if self.allocator.refs[old] > 1:          # shared: copy before writing
                fresh = self.allocator.allocate()
                pairs.append((old, fresh))
                self.allocator.release(old)
                table[i] = fresh
        while len(table) < need:
            table.append(self.allocator.allocate())
        return pairs

    def slot(self, seq, pos: int) -> int:
        """Slot of logical position ``pos``: physical block table[pos // b] at
        offset pos % b ([P1] "Paging"), encoded as block * b + offset."""
        table = self.tables[seq]
        return table[pos // self.block_size] * self.block_size + pos % self.block_size

    def advance(self, seq, n: int) -> None:
        """Commit ``n`` written tokens ([P1] update: length = last position + 1)."""
        self.lengths[seq] += int(n)

    def fork(self, parent, child) -> None:
        """Child aliases the parent's blocks ([P1] "Sharing blocks")."""
        self.create(child)
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for block in self.tables[child]:
            self.allocator.share(block)

    def free(self, seq) -> None:
        for block in self.tables.pop(seq):
            self.allocator.release(block)
        self.lengths.pop(seq)

    def truncate(self, seq, length: int) -> None:
        keep = self.blocks_needed(length)
        for block in self.tables[seq][keep:]:
            self.allocator.release(block)
        del self.tables[seq][keep:]
        self.lengths[seq] = int(length)

    def batch(self, seqs):
        """Block-table rows padded with 0 to the longest table, and lengths
        ([P1] set_batch)."""
        seqs = list(seqs)
        width = max([len(self.tables[s]) for s in seqs] + [1])
        rows = [self.tables[s] + [0] * (width - len(self.tables[s])) for s in seqs]
        return rows, [self.lengths[s] for s in seqs]


class PrefixTable:
    """Prefix cache that only edits block tables and refcounts ([P1] "Prefix caching").

    Keys are whole token prefixes up to the end of a full block; the cache holds
    its own reference on each cached block; eviction is least-recently-used
    among entries nobody else uses.
    """

    def __init__(self, tables: SeqTables):
        self.tables = tables
        self.entries: OrderedDict = OrderedDict()

    def attach(self, seq, prompt) -> int:
        t = self.tables
        t.create(seq)
        size, reused = t.block_size, 0
        prompt = list(prompt)
        # at least one prompt token is always left to prefill
        while reused + size <= len(prompt) - 1:
            key = tuple(prompt[:reused + size])
            block = self.entries.get(key)
            if block is None:
                break
            self.entries.move_to_end(key)
            t.allocator.share(block)
            t.tables[seq].append(block)
            reused += size
        t.lengths[seq] = reused
        return reused

    def remember(self, seq, tokens) -> None:
        t = self.tables
        tokens = list(tokens)
        for index in range(len(tokens) // t.block_size):
            key = tuple(tokens[:(index + 1) * t.block_size])
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
