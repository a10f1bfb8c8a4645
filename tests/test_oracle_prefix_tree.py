"""Pins of the block prefix tree oracle (the radix-tree form of the prefix cache; CPU only).

What fixes it: [P1]'s worked example numbers ("Prefix caching": eight requests
over a 96-token system prompt); exact agreement with the flat prefix table --
the pages' own definition of the cache -- on every trace that evicts nothing
(the two differ only in which entries eviction may drop); and, with evictions,
the invariants the tree must keep (prefix-closed, holder counts equal holders,
free + live = N) plus a hand-worked case where the two policies part ways.
"""
import numpy as np
import pytest

from oracle import blocks
from oracle import prefix_tree as pt
from tests.conftest import golden


def _fill(t, seq, n):
    t.reserve(seq, n)
    t.advance(seq, n)


def _check_invariants(t, tree):
    N = t.allocator.num_blocks
    counts = [0] * N
    for table in t.tables.values():
        for blk in table:
            counts[blk] += 1
    nodes = tree.nodes()
    for n in nodes:
        counts[n.block] += 1
        assert n.parent is tree.root or n.parent in nodes          # prefix-closed
        assert n.parent.children[n.label] is n
    assert counts == t.allocator.refs
    live = sum(1 for c in counts if c > 0)
    assert live + t.allocator.num_free == N
    assert all(counts[blk] == 0 for blk in t.allocator.free)


def test_p1_worked_example_through_the_tree():
    g = golden("p1_prefix_cache.json")
    e, b = g["expected"], g["block_size"]
    t = blocks.SeqTables(256, b)
    tree = pt.BlockPrefixTree(t)
    shared = list(range(1000, 1000 + g["shared_tokens"]))
    prompt_tokens = prefilled = 0
    for r in range(g["requests"]):
        prompt = shared + [r * 100 + i for i in range(g["own_tokens"])]
        reused = tree.attach(r, prompt)
        n = len(prompt) - reused
        _fill(t, r, n)
        tree.remember(r, prompt)
        prompt_tokens += len(prompt)
        prefilled += n
    assert prompt_tokens == e["prompt_tokens"]
    assert prefilled == e["tokens_prefilled"]
    assert 256 - t.allocator.num_free == e["blocks_in_use"]
    # the six shared blocks form one chain; each request's partial seventh block is not cached
    assert len(tree.nodes()) == 6 and len(tree.root.children) == 1
    _check_invariants(t, tree)


def test_at_least_one_prompt_token_is_left_to_prefill():
    t = blocks.SeqTables(16, 4)
    tree = pt.BlockPrefixTree(t)
    tree.attach("a", list(range(8)))
    _fill(t, "a", 8)
    tree.remember("a", list(range(8)))                 # two full blocks cached
    assert tree.attach("b", list(range(8))) == 4       # a whole-block prompt reuses all but its last block
    assert tree.attach("c", list(range(9))) == 8
    assert tree.attach("d", []) == 0 and tree.attach("e", [0]) == 0


def test_remember_descends_through_an_existing_prefix():
    """A sequence that computed a cached prefix into its own blocks (it did not attach)
    adds only its new blocks, under the cached path."""
    t = blocks.SeqTables(16, 2)
    tree = pt.BlockPrefixTree(t)
    tree.attach("a", [1, 2, 3, 4, 9])
    _fill(t, "a", 5)
    tree.remember("a", [1, 2, 3, 4, 9])
    t.create("b")
    _fill(t, "b", 6)
    tree.remember("b", [1, 2, 3, 4, 5, 6])
    a12 = tree.root.children[(1, 2)]
    assert a12.block == t.tables["a"][0] and a12.children[(3, 4)].block == t.tables["a"][1]
    assert a12.children[(3, 4)].children[(5, 6)].block == t.tables["b"][2]
    assert len(tree.nodes()) == 3
    _check_invariants(t, tree)


def test_eviction_takes_leaves_where_the_flat_table_strands_a_prefix():
    """Request "a" caches two blocks; request "b" reuses both (its walk touches the shorter
    prefix first, so the shorter is the older).  After both finish, a request for one free
    block: the flat table drops its least recently used entry -- the first block -- and the
    second becomes unreachable; the tree drops the least recently used leaf, the second
    block, and keeps the first."""
    def run(make):
        t = blocks.SeqTables(6, 2)
        c = make(t)
        for seq, prompt in (("a", [1, 2, 3, 4, 0]), ("b", [1, 2, 3, 4, 9])):
            c.attach(seq, prompt)
            _fill(t, seq, len(prompt) - t.lengths[seq])
            c.remember(seq, prompt)
        assert t.tables["b"][:2] == t.tables["a"][:2]
        t.free("a")
        t.free("b")
        assert t.allocator.num_free == 4
        c.evict(5)
        assert t.allocator.num_free == 5
        return t, c

    t, flat = run(blocks.PrefixTable)
    assert list(flat.entries) == [(1, 2, 3, 4)]                     # the first block went
    assert flat.attach("c", [1, 2, 3, 4, 7]) == 0                   # and the second is unreachable
    t, tree = run(pt.BlockPrefixTree)
    assert [n.label for n in tree.nodes()] == [(1, 2)]              # the leaf went
    assert tree.attach("c", [1, 2, 3, 4, 7]) == 2
    _check_invariants(t, tree)


def test_a_parent_becomes_a_candidate_after_its_last_child():
    t = blocks.SeqTables(4, 2)
    tree = pt.BlockPrefixTree(t)
    tree.attach("a", [1, 2, 3, 4, 5])
    _fill(t, "a", 5)
    tree.remember("a", [1, 2, 3, 4, 5])
    t.free("a")
    tree.evict(4)                               # the leaf, then its parent
    assert tree.nodes() == [] and t.allocator.num_free == 4
    _check_invariants(t, tree)


def test_held_leaves_stay():
    t = blocks.SeqTables(8, 2)
    tree = pt.BlockPrefixTree(t)
    tree.attach("a", [1, 2, 3, 4, 5])
    _fill(t, "a", 5)
    tree.remember("a", [1, 2, 3, 4, 5])
    tree.evict(8)
    assert len(tree.nodes()) == 2                # "a" still holds both blocks
    _check_invariants(t, tree)


# ------------------------------------------------------- traces

def make_trace(seed, n_ops=300, b=4, alphabet=3, evictions=True):
    """Ops over prompts built from a few block texts, so prefixes branch and recur."""
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
            ops.append(("attach", uid, prompt, int(r.integers(0, 2 * b))))
            live.append(uid)
            uid += 1
        elif x < 0.85 or not evictions:
            ops.append(("free", live.pop(int(r.integers(len(live))))))
        else:
            ops.append(("evict", int(r.integers(0, 48))))
    return ops


def replay(ops, make_cache, N=48, b=4, check=None):
    """State after every op: (reused or status, tables, refcounts, free list, cached blocks)."""
    t = blocks.SeqTables(N, b)
    c = make_cache(t)
    states = []
    for op in ops:
        res = None
        if op[0] == "attach":
            _, seq, prompt, gen = op
            res = c.attach(seq, prompt)
            need = len(prompt) - res + gen
            if t.blocks_needed(t.lengths[seq] + need) - len(t.tables[seq]) > t.allocator.num_free:
                c.evict(t.blocks_needed(t.lengths[seq] + need) - len(t.tables[seq]))
            try:
                _fill(t, seq, need)
                c.remember(seq, list(prompt) + [7] * gen)
            except MemoryError:
                res = "oom"
        elif op[0] == "free":
            if op[1] in t.tables:
                t.free(op[1])
        else:
            c.evict(op[1])
        if check:
            check(t, c)
        cached = sorted(c.entries.values()) if hasattr(c, "entries") else c.cached_blocks()
        states.append((res, {k: list(v) for k, v in t.tables.items()}, list(t.allocator.refs),
                       list(t.allocator.free), cached))
    return states


@pytest.mark.parametrize("seed", range(6))
def test_tree_equals_flat_table_when_nothing_is_evicted(seed):
    ops = make_trace(seed, evictions=False)
    want = replay(ops, blocks.PrefixTable, N=4096)
    got = replay(ops, pt.BlockPrefixTree, N=4096, check=_check_invariants)
    assert got == want
    reused = [s[0] for s in want if isinstance(s[0], int)]
    assert max(reused) >= 8 and sum(x > 0 for x in reused) >= 10


@pytest.mark.parametrize("seed", range(6))
def test_tree_invariants_hold_on_traces_with_eviction(seed):
    states = replay(make_trace(seed), pt.BlockPrefixTree, check=_check_invariants)
    # the trace reuses prefixes, evicts and runs out of blocks
    reused = [s[0] for s in states if isinstance(s[0], int)]
    assert sum(x > 0 for x in reused) >= 10
    assert sum(len(b[4]) < len(a[4]) for a, b in zip(states, states[1:])) >= 5
    assert any(s[0] == "oom" for s in states)
