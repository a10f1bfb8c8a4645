"""Host bookkeeping of the paged KV cache: pool, block tables, prefix index.

TEST INFRASTRUCTURE (oracle): restated from [P1] "25. Paged attention and
prefix caching", sections "Paging", "The allocator", "The paged cache",
"Sharing blocks: forks and copy-on-write" and "Prefix caching".  What the
pages fix, and what every structure below keeps true after each operation:

  * Pool: every physical block is either free (holder count 0, on the free
    queue exactly once) or live (count = number of block-table entries plus
    prefix-index entries that hold it).  free + live = N at all times.
  * A sequence of L tokens holds ceil(L / b) blocks; logical position p lives
    in the table's entry p // b at offset p % b ("Paging").
  * A block with more than one holder is never written: before tokens land in
    it, the writer gets a private copy (copy-on-write, "Sharing blocks").
  * The prefix index maps the key of a full block's prefix to the block; it
    holds a reference of its own, and reclaims least-recently-used entries
    whose block no sequence holds ("Prefix caching").

Readings where the pages differ or are silent:
  * free-queue order: first-in first-out ([P1] "The allocator"), seeded with
    a caller-given initial order ([P2] "Код" takes the end of a list instead);
  * over-release: checked before the count changes; RuntimeError, state
    unchanged ([P2] "Код"; [P1] would leave the count at -1);
  * sharing a free block (count 0) is a caller bug: RuntimeError;
  * a reservation that cannot be met raises MemoryError before any state
    changes (all-or-nothing; [P1] raises part-way through);
  * no zeroing of a block when it is handed out ([P2] zeroes; [P1] does not).
"""
from __future__ import annotations

from collections import OrderedDict, deque


class BlockAllocator:
    """N physical blocks: a FIFO queue of the free ones and a holder count per block."""

    def __init__(self, num_blocks: int, order=None):
        n = int(num_blocks)
        first_free = list(range(n)) if order is None else [int(x) for x in order]
        if sorted(first_free) != list(range(n)):
            raise ValueError("initial order must be a permutation of the pool")
        self.num_blocks = n
        self.refs = [0] * n             # holder count per block; 0 <=> on the free queue
        self.free = deque(first_free)   # the block free the longest is at the left

    @property
    def num_free(self) -> int:
        return len(self.free)

    def _require_live(self, block: int, what: str) -> None:
        if self.refs[block] < 1:
            raise RuntimeError(f"{what}: block {block} has no holder")

    def allocate(self) -> int:
        """Hand out the block that has been free the longest, with one holder."""
        if len(self.free) == 0:
            raise MemoryError("KV block pool exhausted")
        block = self.free.popleft()
        self.refs[block] = 1
        return block

    def share(self, block: int) -> None:
        """One more holder of a live block."""
        self._require_live(block, "share")
        self.refs[block] = self.refs[block] + 1

    def release(self, block: int) -> None:
        """One holder fewer; the last one returns the block to the back of the queue."""
        self._require_live(block, "release (more releases than references)")
        left = self.refs[block] - 1
        self.refs[block] = left
        if left == 0:
            self.free.append(block)


class SeqTables:
    """Block table and length of every live sequence, over one pool.

    Copy-on-write is reported, not performed: ``reserve`` returns the (source,
    destination) block pairs the device must copy in every layer's K and V
    pools before it writes.
    """

    def __init__(self, num_blocks: int, block_size: int, order=None):
        self.allocator = BlockAllocator(num_blocks, order)
        self.block_size = int(block_size)
        self.tables: dict = {}     # sequence id -> list of physical blocks
        self.lengths: dict = {}    # sequence id -> tokens written

    def blocks_needed(self, tokens: int) -> int:
        """ceil(tokens / b): the blocks that hold ``tokens`` tokens ([P1] "Paging")."""
        q, r = divmod(int(tokens), self.block_size)
        return q + (1 if r else 0)

    def create(self, seq) -> None:
        if seq in self.tables:
            raise ValueError(f"sequence {seq} already exists")
        self.tables[seq], self.lengths[seq] = [], 0

    def reserve(self, seq, new_tokens: int) -> list:
        """Make positions [length, length + new_tokens) writable by ``seq``.

        Two kinds of table entries are touched, in this order ([P1] "The paged
        cache", reserve): existing entries of the written range whose block
        has another holder each get a fresh block (take a fresh block, record
        the copy, drop this sequence's hold on the old one, repoint); then
        fresh blocks are appended until the table covers the range.  The
        whole demand is counted first, so a failure changes nothing.
        """
        table = self.tables[seq]
        length = self.lengths[seq]
        covered = self.blocks_needed(length + int(new_tokens))
        written = range(length // self.block_size, min(covered, len(table)))
        refs = self.allocator.refs
        shared = [i for i in written if refs[table[i]] > 1]
        appended = max(0, covered - len(table))
        if len(shared) + appended > self.allocator.num_free:
            raise MemoryError("KV block pool exhausted")
        copies = []
        for i in shared:
            old, fresh = table[i], self.allocator.allocate()
            copies.append((old, fresh))
            self.allocator.release(old)
            table[i] = fresh
        table.extend(self.allocator.allocate() for _ in range(appended))
        return copies

    def slot(self, seq, pos: int) -> int:
        """Slot of logical position ``pos``: offset pos % b of block table[pos // b]
        ([P1] "Paging"), encoded as block * b + offset."""
        entry, offset = divmod(int(pos), self.block_size)
        return self.tables[seq][entry] * self.block_size + offset

    def advance(self, seq, n: int) -> None:
        """Count ``n`` more written tokens ([P1] update: length = last position + 1)."""
        self.lengths[seq] = self.lengths[seq] + int(n)

    def fork(self, parent, child) -> None:
        """``child`` starts as an alias of every block of ``parent`` ([P1] "Sharing blocks")."""
        self.create(child)
        inherited = list(self.tables[parent])
        for block in inherited:
            self.allocator.share(block)
        self.tables[child] = inherited
        self.lengths[child] = self.lengths[parent]

    def truncate(self, seq, length: int) -> None:
        """Keep the first ``length`` tokens; blocks past them lose this holder, in table order."""
        table = self.tables[seq]
        keep = self.blocks_needed(length)
        dropped = table[keep:]
        del table[keep:]
        for block in dropped:
            self.allocator.release(block)
        self.lengths[seq] = int(length)

    def free(self, seq) -> None:
        """Drop the sequence: every block it holds loses this holder, in table order."""
        self.truncate(seq, 0)
        del self.tables[seq], self.lengths[seq]

    def batch(self, seqs):
        """Rows of the device block table (padded with block 0 to the widest row)
        and the lengths, for ``seqs`` in order ([P1] set_batch)."""
        seqs = list(seqs)
        width = max([1] + [len(self.tables[s]) for s in seqs])
        rows = [list(self.tables[s]) + [0] * (width - len(self.tables[s])) for s in seqs]
        return rows, [self.lengths[s] for s in seqs]


class KeyedPrefixIndex:
    """Prefix index over one SeqTables, generic in how a full block's key is formed.

    ``block_keys(tokens, salt)`` yields the keys of the full blocks of
    ``tokens`` in order; key i must identify tokens[: (i + 1) * b] (and the
    salt).  ``entries`` maps key -> block, least recently used first.
    """

    def __init__(self, tables: SeqTables):
        self.tables = tables
        self.entries: OrderedDict = OrderedDict()

    def block_keys(self, tokens, salt):
        raise NotImplementedError

    def attach(self, seq, prompt, salt: bytes = b"") -> int:
        """Create ``seq`` holding the longest run of cached full blocks that
        starts the prompt, leaving at least one prompt token to prefill (its
        logits are needed).  Returns the tokens reused."""
        prompt = list(prompt)
        b = self.tables.block_size
        usable = max(0, (len(prompt) - 1) // b)   # full blocks that leave a token over
        hits = []
        for i, key in enumerate(self.block_keys(prompt, salt)):
            if i == usable or key not in self.entries:
                break
            hits.append(key)
        self.tables.create(seq)
        held = []
        for key in hits:
            self.entries.move_to_end(key)          # most recently used now
            block = self.entries[key]
            self.tables.allocator.share(block)
            held.append(block)
        self.tables.tables[seq] = held
        self.tables.lengths[seq] = len(held) * b
        return len(held) * b

    def remember(self, seq, tokens, salt: bytes = b"") -> None:
        """Publish the full blocks of ``seq`` (which holds ``tokens``) whose key
        is not cached yet; the index takes its own reference on each."""
        table = self.tables.tables[seq]
        for i, key in enumerate(self.block_keys(list(tokens), salt)):
            if key in self.entries:
                continue
            self.tables.allocator.share(table[i])
            self.entries[key] = table[i]

    def evict(self, blocks_wanted: int) -> None:
        """Free cached blocks, least recently used first, until ``blocks_wanted``
        blocks are free; only entries whose block has no holder but the index
        are candidates."""
        alloc = self.tables.allocator
        short = int(blocks_wanted) - alloc.num_free
        if short <= 0:
            return
        idle = [key for key, block in self.entries.items() if alloc.refs[block] == 1]
        for key in idle[:short]:
            alloc.release(self.entries.pop(key))


class PrefixTable(KeyedPrefixIndex):
    """[P1]'s prefix cache: a block's key is the whole token tuple up to its end."""

    def block_keys(self, tokens, salt):
        if salt:
            raise ValueError("token-tuple keys carry no salt")
        b = self.tables.block_size
        for end in range(b, len(tokens) + 1, b):
            yield tuple(tokens[:end])
