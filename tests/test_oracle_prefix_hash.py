"""Pins of the hash-chain prefix cache oracle (CPU only).

The chain keys are pinned by what the pages require of them ([P1] "Prefix
caching": the key of a block covers its whole history and whatever else
changes the activations) and by the published SHA-256 examples; the
hash-keyed table is pinned to the tuple-keyed table, which is the pages'
own definition of the cache, on traces where the same block text recurs
under different histories and different salts.
"""
import numpy as np
import pytest

from oracle import blocks
from oracle import prefix_hash as ph
from tests.conftest import golden


def test_sha256_matches_published_examples():
    import hashlib
    for ex in golden("fips180_sha256_examples.json")["examples"]:
        assert hashlib.sha256(ex["message"].encode()).hexdigest() == ex["sha256"]


def test_keys_cover_only_full_blocks_and_extend_by_prefix():
    toks = list(range(100, 139))                        # 39 tokens, b = 8 -> 4 full blocks
    keys = ph.chain_keys(toks, 8, b"m")
    assert len(keys) == 4 and all(len(k) == 32 for k in keys)
    for n in range(0, 40):
        assert ph.chain_keys(toks[:n], 8, b"m") == keys[:n // 8]   # a key never depends on later tokens


def test_same_block_text_under_different_history_differs():
    a = [1, 2, 3, 4, 9, 9, 9, 9]
    b = [5, 6, 7, 8, 9, 9, 9, 9]
    ka, kb = ph.chain_keys(a, 4), ph.chain_keys(b, 4)
    assert ka[0] != kb[0]
    assert ka[1] != kb[1]                               # same text [9, 9, 9, 9], different history
    assert ph.chain_keys([9, 9, 9, 9, 9, 9, 9, 9], 4)[1] != ph.chain_keys([9, 9, 9, 9], 4)[0]


def test_salt_separates_every_key():
    toks = list(range(64))
    base = ph.chain_keys(toks, 16, b"")
    for salt in (b"rev-2", b"lora:7", b"\x00", b"rev-2\x00"):
        other = ph.chain_keys(toks, 16, salt)
        assert not set(base) & set(other)
    assert ph.root_key(b"ab") != ph.root_key(b"a")


def test_token_order_width_and_block_size_matter():
    assert ph.chain_keys([1, 2, 3, 4], 4) != ph.chain_keys([2, 1, 3, 4], 4)
    assert ph.chain_keys([1, 0, 0, 0], 4) != ph.chain_keys([1 + (1 << 32), 0, 0, 0], 4)   # full 64-bit ids
    assert ph.chain_keys([-1, 0, 0, 0], 4) != ph.chain_keys([(1 << 32) - 1, 0, 0, 0], 4)
    assert ph.chain_keys(list(range(8)), 8)[0] != ph.chain_keys(list(range(8)), 4)[1]


def test_p1_worked_example_with_chain_keys():
    g = golden("p1_prefix_cache.json")
    e, b = g["expected"], g["block_size"]
    t = blocks.SeqTables(256, b)
    pc = ph.HashPrefixTable(t)
    shared = list(range(1000, 1000 + g["shared_tokens"]))
    prompt_tokens = prefilled = 0
    for r in range(g["requests"]):
        prompt = shared + [r * 100 + i for i in range(g["own_tokens"])]
        reused = pc.attach(r, prompt, b"model-a")
        n = len(prompt) - reused
        t.reserve(r, n)
        t.advance(r, n)
        pc.remember(r, prompt, b"model-a")
        prompt_tokens += len(prompt)
        prefilled += n
    assert prompt_tokens == e["prompt_tokens"]
    assert prefilled == e["tokens_prefilled"]
    assert 256 - t.allocator.num_free == e["blocks_in_use"]


# ------------------------------------------------------- differential traces

SALTS = (b"", b"rev-2", b"lora:7")


def make_trace(seed, n_ops=250, b=4, alphabet=3):
    """Ops over prompts built from a few block texts, so equal block text recurs
    under different histories; salts vary; frees and evictions interleave."""
    r = np.random.default_rng(seed)
    texts = [[int(x) for x in r.integers(0, 4, size=b)] for _ in range(alphabet)]
    ops, live, uid = [], [], 0
    for _ in range(n_ops):
        x = r.random()
        if x < 0.5 or not live:
            prompt = []
            for _ in range(int(r.integers(0, 6))):
                prompt += texts[int(r.integers(alphabet))]
            prompt += [int(t) for t in r.integers(0, 4, size=int(r.integers(0, b + 1)))]
            gen = int(r.integers(0, 2 * b))
            ops.append(("attach", uid, prompt, SALTS[int(r.integers(len(SALTS)))], gen))
            live.append(uid)
            uid += 1
        elif x < 0.85:
            ops.append(("free", live.pop(int(r.integers(len(live))))))
        else:
            ops.append(("evict", int(r.integers(0, 48))))
    return ops


class TupleWithSalt:
    """The tuple-keyed table with the salt folded into every token of the key."""

    def __init__(self, t):
        self.pc = blocks.PrefixTable(t)

    def attach(self, seq, prompt, salt):
        return self.pc.attach(seq, [(salt, x) for x in prompt])

    def remember(self, seq, tokens, salt):
        self.pc.remember(seq, [(salt, x) for x in tokens])

    def evict(self, n):
        self.pc.evict(n)

    def cached_blocks(self):
        return list(self.pc.entries.values())


class Hashed:
    def __init__(self, t):
        self.pc = ph.HashPrefixTable(t)

    def attach(self, seq, prompt, salt):
        return self.pc.attach(seq, prompt, salt)

    def remember(self, seq, tokens, salt):
        self.pc.remember(seq, tokens, salt)

    def evict(self, n):
        self.pc.evict(n)

    def cached_blocks(self):
        return list(self.pc.entries.values())


def replay(ops, make_cache, N=48, b=4):
    """State after every op: (reused or status, tables, refs, free list, cached blocks in LRU order)."""
    t = blocks.SeqTables(N, b)
    c = make_cache(t)
    states = []
    for op in ops:
        res = None
        if op[0] == "attach":
            _, seq, prompt, salt, gen = op
            res = c.attach(seq, prompt, salt)
            need = len(prompt) - res + gen
            if t.blocks_needed(t.lengths[seq] + need) - len(t.tables[seq]) > t.allocator.num_free:
                c.evict(t.blocks_needed(t.lengths[seq] + need) - len(t.tables[seq]))
            try:
                t.reserve(seq, need)
                t.advance(seq, need)
                c.remember(seq, list(prompt) + [7] * gen, salt)
            except MemoryError:
                res = "oom"
        elif op[0] == "free":
            if op[1] in t.tables:
                t.free(op[1])
        else:
            c.evict(op[1])
        states.append((res, {k: list(v) for k, v in t.tables.items()}, list(t.allocator.refs),
                       list(t.allocator.free), c.cached_blocks()))
    return states


@pytest.mark.parametrize("seed", range(6))
def test_hash_table_equals_tuple_table_on_traces(seed):
    ops = make_trace(seed)
    want = replay(ops, TupleWithSalt)
    got = replay(ops, Hashed)
    assert got == want
    # the trace exercises sharing, evictions that drop entries, and exhaustion
    reused = [s[0] for s in want if isinstance(s[0], int)]
    assert max(reused) >= 8 and sum(x > 0 for x in reused) >= 10
    assert sum(len(b[4]) < len(a[4]) for a, b in zip(want, want[1:])) >= 10
    assert any(s[0] == "oom" for s in want)
