"""The C++ hash-chain prefix table against the oracle (CPU only).

Chain keys must equal the oracle's byte for byte; the table must make the
same decisions (blocks reused, references, least-recently-used order,
evictions) as the oracle's HashPrefixTable on traces where equal block text
recurs under different histories and salts.
"""
import numpy as np
import pytest

from oracle import blocks as oblocks
from oracle import prefix_hash as ph
from paged_kv_cache_66_gb300._lib import PagedKVError
from paged_kv_cache_66_gb300.host import HostBlockManager, prefix_chain_keys, prefix_salt
from tests.test_oracle_prefix_hash import make_trace


@pytest.mark.parametrize("n,b", [(0, 16), (15, 16), (16, 16), (1000, 16), (777, 32), (9, 1)])
def test_chain_keys_match_oracle(n, b):
    r = np.random.default_rng(n * 31 + b)
    toks = r.integers(-(1 << 62), 1 << 62, size=n)
    for salt in (b"", prefix_salt("rev-2", "lora:7", [b"\x00img"]), bytes(range(256)) * 3):
        assert prefix_chain_keys(toks, b, salt) == ph.chain_keys(toks.tolist(), b, salt)


def test_prefix_salt_fields_are_unambiguous():
    assert prefix_salt("ab", "") != prefix_salt("a", "b")
    assert prefix_salt("r", "a", [b"x"]) != prefix_salt("r", "a")
    assert prefix_salt() == prefix_salt("", "")


def test_invalid_arguments():
    h = HostBlockManager(8, 4)
    with pytest.raises(PagedKVError):
        prefix_chain_keys([1, 2, 3, 4], 0)
    assert h.hprefix_attach(1, [1, 2, 3, 4, 5]) == 0
    with pytest.raises(ValueError):
        h.hprefix_attach(1, [1, 2])                        # sequence exists
    with pytest.raises(KeyError):
        h.hprefix_remember(99, [1, 2, 3, 4])
    with pytest.raises(PagedKVError):
        h.hprefix_remember(1, [1, 2, 3, 4])                # holds no block yet


def _replay_cpp(ops, N=48, b=4):
    h = HostBlockManager(N, b)
    live, states = set(), []
    for op in ops:
        res = None
        if op[0] == "attach":
            _, seq, prompt, salt, gen = op
            res = h.hprefix_attach(seq, prompt, salt)
            live.add(seq)
            need = len(prompt) - res + gen
            grow = -(-(h.length(seq) + need) // b) - len(h.table(seq))
            if grow > h.num_free:
                h.hprefix_evict(grow)
            try:
                h.reserve(seq, need)
                h.advance(seq, need)
                h.hprefix_remember(seq, list(prompt) + [7] * gen, salt)
            except MemoryError:
                res = "oom"
        elif op[0] == "free":
            if op[1] in live:
                h.free(op[1])
                live.discard(op[1])
        else:
            h.hprefix_evict(op[1])
        states.append((res, {s: h.table(s) for s in sorted(live)}, [h.refcount(x) for x in range(N)],
                       h.num_free, h.hprefix_blocks()))
    return states


def _replay_oracle(ops, N=48, b=4):
    t = oblocks.SeqTables(N, b)
    pc = ph.HashPrefixTable(t)
    states = []
    for op in ops:
        res = None
        if op[0] == "attach":
            _, seq, prompt, salt, gen = op
            res = pc.attach(seq, prompt, salt)
            need = len(prompt) - res + gen
            grow = t.blocks_needed(t.lengths[seq] + need) - len(t.tables[seq])
            if grow > t.allocator.num_free:
                pc.evict(grow)
            try:
                t.reserve(seq, need)
                t.advance(seq, need)
                pc.remember(seq, list(prompt) + [7] * gen, salt)
            except MemoryError:
                res = "oom"
        elif op[0] == "free":
            if op[1] in t.tables:
                t.free(op[1])
        else:
            pc.evict(op[1])
        states.append((res, {s: list(t.tables[s]) for s in sorted(t.tables)}, list(t.allocator.refs),
                       t.allocator.num_free, list(pc.entries.values())))
    return states


@pytest.mark.parametrize("seed", range(6))
def test_cpp_hash_table_matches_oracle(seed):
    ops = make_trace(seed)
    assert _replay_cpp(ops) == _replay_oracle(ops)


def test_tuple_and_hash_tables_are_separate():
    h = HostBlockManager(16, 4)
    p = list(range(9))
    assert h.hprefix_attach(0, p) == 0
    h.reserve(0, 9)
    h.advance(0, 9)
    h.hprefix_remember(0, p)
    assert h.hprefix_entries == 2 and h.prefix_entries == 0
    assert h.prefix_attach(1, p) == 0                      # the tuple table has no entry
    assert h.hprefix_attach(2, p) == 8
    assert h.hprefix_attach(3, p, salt=prefix_salt("other-revision")) == 0
