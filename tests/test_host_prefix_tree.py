"""The C++ block prefix tree against the oracle's (CPU only).

The tree must make the same decisions as the oracle's BlockPrefixTree op for
op -- blocks reused, tables, holder counts, free blocks, the cached blocks --
on traces where prefixes branch and recur and leaves are evicted.
"""
import pytest

from oracle import blocks as oblocks
from oracle import prefix_tree as opt
from paged_kv_cache_66_gb300._lib import PagedKVError
from paged_kv_cache_66_gb300.host import HostBlockManager
from tests.conftest import golden
from tests.test_oracle_prefix_tree import make_trace


def _replay_cpp(ops, N=48, b=4):
    h = HostBlockManager(N, b)
    live, states = set(), []
    for op in ops:
        res = None
        if op[0] == "attach":
            _, seq, prompt, gen = op
            res = h.tprefix_attach(seq, prompt)
            live.add(seq)
            need = len(prompt) - res + gen
            grow = -(-(h.length(seq) + need) // b) - len(h.table(seq))
            if grow > h.num_free:
                h.tprefix_evict(grow)
            try:
                h.reserve(seq, need)
                h.advance(seq, need)
                h.tprefix_remember(seq, list(prompt) + [7] * gen)
            except MemoryError:
                res = "oom"
        elif op[0] == "free":
            if op[1] in live:
                h.free(op[1])
                live.discard(op[1])
        else:
            h.tprefix_evict(op[1])
        states.append((res, {s: h.table(s) for s in sorted(live)}, [h.refcount(x) for x in range(N)],
                       h.num_free, h.tprefix_blocks(), h.tprefix_nodes))
    return states


def _replay_oracle(ops, N=48, b=4):
    t = oblocks.SeqTables(N, b)
    tree = opt.BlockPrefixTree(t)
    states = []
    for op in ops:
        res = None
        if op[0] == "attach":
            _, seq, prompt, gen = op
            res = tree.attach(seq, prompt)
            need = len(prompt) - res + gen
            grow = t.blocks_needed(t.lengths[seq] + need) - len(t.tables[seq])
            if grow > t.allocator.num_free:
                tree.evict(grow)
            try:
                t.reserve(seq, need)
                t.advance(seq, need)
                tree.remember(seq, list(prompt) + [7] * gen)
            except MemoryError:
                res = "oom"
        elif op[0] == "free":
            if op[1] in t.tables:
                t.free(op[1])
        else:
            tree.evict(op[1])
        cached = tree.cached_blocks()
        states.append((res, {s: list(t.tables[s]) for s in sorted(t.tables)}, list(t.allocator.refs),
                       t.allocator.num_free, cached, len(cached)))
    return states


@pytest.mark.parametrize("seed", range(8))
def test_cpp_tree_matches_oracle(seed):
    ops = make_trace(seed)
    want = _replay_oracle(ops)
    assert _replay_cpp(ops) == want
    assert sum(len(b[4]) < len(a[4]) for a, b in zip(want, want[1:])) >= 5   # evictions happened


@pytest.mark.parametrize("seed", range(3))
def test_cpp_tree_matches_oracle_on_a_larger_pool(seed):
    ops = make_trace(100 + seed, n_ops=600, b=2, alphabet=4)
    assert _replay_cpp(ops, N=200, b=2) == _replay_oracle(ops, N=200, b=2)


def test_cpp_tree_p1_worked_example():
    g = golden("p1_prefix_cache.json")
    e, b = g["expected"], g["block_size"]
    h = HostBlockManager(256, b)
    shared = list(range(1000, 1000 + g["shared_tokens"]))
    prompt_tokens = prefilled = 0
    for r in range(g["requests"]):
        prompt = shared + [r * 100 + i for i in range(g["own_tokens"])]
        reused = h.tprefix_attach(r, prompt)
        n = len(prompt) - reused
        h.reserve(r, n)
        h.advance(r, n)
        h.tprefix_remember(r, prompt)
        prompt_tokens += len(prompt)
        prefilled += n
    assert (prompt_tokens, prefilled, 256 - h.num_free) == (e["prompt_tokens"], e["tokens_prefilled"],
                                                          e["blocks_in_use"])
    assert h.tprefix_nodes == 6


def test_invalid_arguments_and_independence():
    h = HostBlockManager(16, 4)
    p = list(range(9))
    assert h.tprefix_attach(0, p) == 0
    with pytest.raises(ValueError):
        h.tprefix_attach(0, p)                             # sequence exists
    with pytest.raises(KeyError):
        h.tprefix_remember(99, p)
    with pytest.raises(PagedKVError):
        h.tprefix_remember(0, p)                           # holds no block yet
    h.reserve(0, 9)
    h.advance(0, 9)
    h.tprefix_remember(0, p)
    assert h.tprefix_nodes == 2 and h.prefix_entries == 0 and h.hprefix_entries == 0
    assert h.prefix_attach(1, p) == 0 and h.hprefix_attach(2, p) == 0   # the other tables see nothing
    assert h.tprefix_attach(3, p) == 8
