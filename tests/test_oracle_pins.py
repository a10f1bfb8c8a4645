"""Pins of the oracle to what the pages and mathematics fix (CPU only).

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/*.json, each with its citation), closed forms,
brute force on tiny inputs, or an independent library routine (torch's
scaled_dot_product_attention in fp64).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, blocks, cache_ops
from tests.conftest import golden


# ------------------------------------------------------------------ slots & blocks

def test_slot_worked_example():
    g = golden("p1_slot_example.json")
    t = blocks.SeqTables(num_blocks=8, block_size=g["block_size"])
    t.create("s")
    t.tables["s"] = list(g["table"])
    t.lengths["s"] = len(g["table"]) * g["block_size"]
    slot = t.slot("s", g["position"])
    assert divmod(slot, g["block_size"]) == tuple(g["expected_block_offset"])
    assert g["position"] // g["block_size"] == g["expected_logical_block"]


@pytest.mark.parametrize("b", [1, 4, 16, 32])
def test_blocks_needed_and_waste_bruteforce(b):
    t = blocks.SeqTables(num_blocks=1, block_size=b)
    for L in range(0, 300):
        n = t.blocks_needed(L)
        # brute force: smallest n with n * b >= L
        brute = next(k for k in range(0, L + 2) if k * b >= L)
        assert n == brute
        assert 0 <= n * b - L < b


def test_utilization_demo_arithmetic():
    g = golden("p1_utilization_demo.json")
    p, b = g["printed"], g["block_size"]
    assert p["static_slots_reserved"] == p["requests"] * g["static_slot_tokens"]
    assert p["paged_slots_reserved"] % b == 0
    # waste at most b-1 slots per sequence ([P1] "Paging")
    assert 0 <= p["paged_slots_reserved"] - p["tokens_stored"] <= p["requests"] * (b - 1)
    assert round(p["tokens_stored"] / p["static_slots_reserved"], 3) == p["static_utilization"]
    assert round(p["tokens_stored"] / p["paged_slots_reserved"], 3) == p["paged_utilization"]


def test_bytes_model():
    g = golden("p2_bytes_model.json")
    e = g["expected"]
    per_tok_layer = 2 * g["kv_heads"] * g["head_dim"] * g["elt_bytes"]
    assert per_tok_layer == e["bytes_per_token_per_layer"]
    assert per_tok_layer * g["layers"] == e["bytes_per_token_all_layers"]
    assert per_tok_layer * g["layers"] * g["block_size"] == e["bytes_per_block_all_layers"]
    assert per_tok_layer * g["layers"] * 4096 == e["bytes_at_4k"]
    assert per_tok_layer * g["layers"] * 32768 == e["bytes_at_32k"]
    t = blocks.SeqTables(1, g["block_size"])
    assert t.blocks_needed(32768) * 4 == e["table_bytes_at_32k_int32"]
    # one (block, kv head) tile of K in the [N, Hkv, b, D] pool is contiguous
    pool = cache_ops.new_pool(4, g["kv_heads"], g["block_size"], g["head_dim"], torch.float16)
    tile = pool[1, 3]
    assert tile.is_contiguous() and tile.numel() * 2 == e["head_block_bytes"]


# ------------------------------------------------------------------ allocator

def test_allocator_fifo_and_refcounts():
    order = [3, 0, 2, 1]
    a = blocks.BlockAllocator(4, order)
    got = [a.allocate() for _ in range(4)]
    assert got == order
    with pytest.raises(MemoryError):
        a.allocate()
    a.share(2)
    a.release(2)
    assert a.num_free == 0          # still referenced once
    a.release(2)
    assert a.num_free == 1 and list(a.free) == [2]
    a.release(0)
    assert list(a.free) == [2, 0]   # released blocks go to the tail
    assert a.allocate() == 2


def test_over_release_raises_and_keeps_state():
    a = blocks.BlockAllocator(2)
    blk = a.allocate()
    a.release(blk)
    before = (list(a.free), list(a.refs))
    with pytest.raises(RuntimeError):
        a.release(blk)
    assert (list(a.free), list(a.refs)) == before
    with pytest.raises(RuntimeError):
        a.share(blk)


def test_duplicate_create_raises():
    t = blocks.SeqTables(4, 4)
    t.create(1)
    with pytest.raises(ValueError):
        t.create(1)


def test_reserve_exhaustion_is_all_or_nothing():
    t = blocks.SeqTables(4, 4)
    t.create(0)
    t.reserve(0, 8)
    t.advance(0, 8)
    t.create(1)
    state = ([list(x) for x in t.tables.values()], dict(t.lengths), list(t.allocator.free),
             list(t.allocator.refs))
    with pytest.raises(MemoryError):
        t.reserve(1, 12)            # needs 3 blocks, 2 free
    assert state == ([list(x) for x in t.tables.values()], dict(t.lengths),
                     list(t.allocator.free), list(t.allocator.refs))


def _check_invariants(t: blocks.SeqTables, extra_refs=()):
    N = t.allocator.num_blocks
    counts = [0] * N
    for table in t.tables.values():
        for blk in table:
            counts[blk] += 1
    for blk in extra_refs:
        counts[blk] += 1
    assert counts == t.allocator.refs
    live = sum(1 for c in counts if c > 0)
    assert live + t.allocator.num_free == N
    assert sorted(set(t.allocator.free)) == sorted(t.allocator.free)
    assert all(counts[blk] == 0 for blk in t.allocator.free)
    for s, table in t.tables.items():
        assert len(table) == t.blocks_needed(t.lengths[s])


def test_random_op_invariants():
    r = np.random.default_rng(0)
    t = blocks.SeqTables(64, 4, r.permutation(64))
    live = []
    nxt = 0
    for _ in range(2000):
        op = r.integers(0, 5)
        try:
            if op == 0 or not live:
                t.create(nxt)
                live.append(nxt)
                nxt += 1
            elif op == 1:
                s = live[r.integers(len(live))]
                n = int(r.integers(1, 9))
                t.reserve(s, n)
                t.advance(s, n)
            elif op == 2:
                s = live[r.integers(len(live))]
                t.fork(s, nxt)
                live.append(nxt)
                nxt += 1
            elif op == 3:
                s = live.pop(r.integers(len(live)))
                t.free(s)
            else:
                s = live[r.integers(len(live))]
                t.truncate(s, int(r.integers(0, t.lengths[s] + 1)))
        except MemoryError:
            pass
        _check_invariants(t)


# ------------------------------------------------------------------ fork / CoW / prefix

def _fill(t, seq, n):
    pairs = t.reserve(seq, n)
    t.advance(seq, n)
    return pairs


def test_fork_cow_p1_numbers():
    g = golden("p1_fork_cow.json")
    t = blocks.SeqTables(64, g["block_size"])
    t.create("p")
    _fill(t, "p", g["prompt_tokens"])
    used0 = 64 - t.allocator.num_free
    for i in range(g["forks"]):
        t.fork("p", f"c{i}")
    used1 = 64 - t.allocator.num_free
    pairs = []
    for i in range(g["forks"]):
        pairs += _fill(t, f"c{i}", 1)
    used2 = 64 - t.allocator.num_free
    e = g["expected"]
    assert used0 == e["parent_blocks"]
    assert used1 - used0 == e["new_blocks_after_4_forks"]
    assert used2 - used1 == e["new_blocks_after_each_sample_writes_a_token"]
    # every copy duplicates the shared partial last block of the prompt
    assert len(pairs) == g["forks"]
    assert all(src == t.tables["p"][-1] for src, _ in pairs)
    _check_invariants(t)


def test_prefix_sharing_p2_numbers():
    g = golden("p2_prefix_sharing.json")
    e, b = g["expected"], g["block_size"]
    t = blocks.SeqTables(1024, b)
    t.create("base")
    _fill(t, "base", g["system_prompt_tokens"])
    assert len(t.tables["base"]) == e["prompt_blocks"]
    for i in range(g["forks"]):
        t.fork("base", i)
        for _ in range(g["tokens_per_fork"]):
            _fill(t, i, 1)
    used = 1024 - t.allocator.num_free
    shared = set(t.tables[0]) & set(t.tables[1])
    no_share = g["forks"] * t.blocks_needed(g["system_prompt_tokens"] + g["tokens_per_fork"])
    c = g["bytes_per_block_config"]
    block_bytes = 2 * c["layers"] * b * c["kv_heads"] * c["head_dim"] * c["elt_bytes"]
    assert len(shared) == e["shared_blocks"]
    assert t.tables[0][-1] != t.tables[1][-1]
    assert used == e["blocks_used"]
    assert no_share == e["blocks_without_sharing"]
    assert no_share - used == e["blocks_saved"]
    assert (no_share - used) * block_bytes // 2**20 == e["mib_saved"]
    t.free("base")
    assert 1024 - t.allocator.num_free == e["used_after_base_free"]
    for i in range(g["forks"]):
        t.free(i)
    assert 1024 - t.allocator.num_free == e["used_after_all_free"]


def test_prefix_cache_p1_numbers():
    g = golden("p1_prefix_cache.json")
    e, b = g["expected"], g["block_size"]
    t = blocks.SeqTables(256, b)
    pc = blocks.PrefixTable(t)
    shared = list(range(1000, 1000 + g["shared_tokens"]))
    prompt_tokens = prefilled = 0
    for r in range(g["requests"]):
        prompt = shared + [r * 100 + i for i in range(g["own_tokens"])]
        reused = pc.attach(r, prompt)
        n = len(prompt) - reused
        _fill(t, r, n)
        pc.remember(r, prompt)
        prompt_tokens += len(prompt)
        prefilled += n
    assert prompt_tokens == e["prompt_tokens"]
    assert prefilled == e["tokens_prefilled"]
    assert 256 - t.allocator.num_free == e["blocks_in_use"]
    assert g["requests"] * t.blocks_needed(g["shared_tokens"] + g["own_tokens"]) == \
        e["blocks_without_sharing"]
    _check_invariants(t, extra_refs=list(pc.entries.values()))


def test_prefix_cache_evict_lru_only_unused():
    t = blocks.SeqTables(8, 2)
    pc = blocks.PrefixTable(t)
    pc.attach("a", [1, 2, 3, 4, 5])
    _fill(t, "a", 5)
    pc.remember("a", [1, 2, 3, 4, 5])        # caches 2 full blocks
    assert len(pc.entries) == 2
    pc.evict(8)                               # all referenced by "a": nothing evicted
    assert len(pc.entries) == 2
    t.free("a")
    pc.evict(t.allocator.num_free + 1)        # evicts the least recently used first
    assert len(pc.entries) == 1 and list(pc.entries)[0] == (1, 2, 3, 4)
    _check_invariants(t, extra_refs=list(pc.entries.values()))


def test_fragmentation_p2():
    g = golden("p2_fragmentation.json")
    e, b = g["expected"], g["block_size"]
    lengths = np.random.default_rng(g["seed"]).integers(g["low"], g["high_inclusive"] + 1,
                                                        size=g["sequences"])
    t = blocks.SeqTables(100_000, b)
    for i, L in enumerate(lengths):
        t.create(i)
        for _ in range(int(L)):             # token-by-token growth, allocate on demand
            _fill(t, i, 1)
    paged = 100_000 - t.allocator.num_free
    reserved = g["sequences"] * (g["max_len"] // b)
    waste = paged * b - int(lengths.sum())
    assert reserved == e["reserved_blocks"]
    assert waste / (paged * b) < e["waste_ratio_below"]
    assert paged < e["paged_over_reserved_below"] * reserved


# ------------------------------------------------------------------ append / copy

def test_append_gather_roundtrip_scrambled():
    r = np.random.default_rng(5)
    b, Hkv, D, N = 4, 2, 3, 32
    t = blocks.SeqTables(N, b, r.permutation(N))
    pk = cache_ops.new_pool(N, Hkv, b, D, torch.float32)
    pv = cache_ops.new_pool(N, Hkv, b, D, torch.float32)
    rows = {}
    for s, L in enumerate([1, 3, 4, 5, 9]):
        t.create(s)
        t.reserve(s, L)
        k = torch.tensor(r.normal(size=(L, Hkv, D)), dtype=torch.float32)
        v = torch.tensor(r.normal(size=(L, Hkv, D)), dtype=torch.float32)
        slots = [t.slot(s, p) for p in range(L)]
        cache_ops.append(pk, pv, k, v, slots, b)
        t.advance(s, L)
        rows[s] = (k, v)
    for s, (k, v) in rows.items():
        L = t.lengths[s]
        K = attention.gather_history(pk, t.tables[s], L, b)
        V = attention.gather_history(pv, t.tables[s], L, b)
        assert np.array_equal(K, k.double().numpy())
        assert np.array_equal(V, v.double().numpy())


def test_append_negative_slot_skipped():
    pk = cache_ops.new_pool(2, 1, 2, 2, torch.float32)
    pv = cache_ops.new_pool(2, 1, 2, 2, torch.float32)
    k = torch.ones(2, 1, 2)
    cache_ops.append(pk, pv, k, k, [-1, 3], 2)
    assert pk[1, 0, 1].tolist() == [1.0, 1.0] and pk.sum().item() == 2.0


def test_cow_keeps_parent_history():
    """Mutate-after-fork must not clobber the peer ([P1] milestone test, [P4]
    functional checks): the parent's bytes are unchanged after the child writes."""
    r = np.random.default_rng(9)
    b, Hkv, D, N, layers = 4, 2, 4, 16, 3
    t = blocks.SeqTables(N, b, r.permutation(N))
    K = [cache_ops.new_pool(N, Hkv, b, D, torch.float16) for _ in range(layers)]
    V = [cache_ops.new_pool(N, Hkv, b, D, torch.float16) for _ in range(layers)]
    t.create("p")
    t.reserve("p", 6)
    for layer in range(layers):
        x = torch.tensor(r.normal(size=(6, Hkv, D)), dtype=torch.float16)
        cache_ops.append(K[layer], V[layer], x, -x, [t.slot("p", i) for i in range(6)], b)
    t.advance("p", 6)
    before = [attention.gather_history(K[x], t.tables["p"], 6, b) for x in range(layers)]
    t.fork("p", "c")
    pairs = t.reserve("c", 1)
    assert len(pairs) == 1 and pairs[0][0] == t.tables["p"][1]
    cache_ops.copy_blocks(K, V, pairs)
    src, dst = pairs[0]
    for layer in range(layers):
        assert torch.equal(K[layer][dst], K[layer][src])
        assert torch.equal(V[layer][dst], V[layer][src])
        y = torch.full((1, Hkv, D), 7.0, dtype=torch.float16)
        cache_ops.append(K[layer], V[layer], y, y, [t.slot("c", 6)], b)
    t.advance("c", 1)
    for layer in range(layers):
        assert np.array_equal(before[layer],
                              attention.gather_history(K[layer], t.tables["p"], 6, b))
        Kc = attention.gather_history(K[layer], t.tables["c"], 7, b)
        assert np.array_equal(Kc[:6], before[layer]) and np.all(Kc[6] == 7.0)


# ------------------------------------------------------------------ attention

def _sdpa(q, K, V, scale):
    """torch's fp64 SDPA with contiguous GQA grouping (repeat_interleave)."""
    Hq, Hkv = q.shape[0], K.shape[1]
    G = Hq // Hkv
    qt = torch.tensor(q, dtype=torch.float64)[:, None, :]          # [Hq, 1, D]
    Kt = torch.tensor(K, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)
    Vt = torch.tensor(V, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("Hq,Hkv,D,L", [(4, 2, 8, 40), (4, 4, 16, 1), (8, 2, 32, 15),
                                          (8, 2, 32, 16), (8, 2, 32, 17), (32, 8, 64, 300),
                                          (8, 1, 128, 97)])
def test_attention_matches_library_sdpa(Hq, Hkv, D, L):
    r = np.random.default_rng(Hq * 1000 + L)
    q = r.normal(size=(Hq, D))
    K = r.normal(size=(L, Hkv, D))
    V = r.normal(size=(L, Hkv, D))
    scale = 1 / math.sqrt(D)
    got = attention.decode_attention(q, K, V, scale)
    np.testing.assert_allclose(got, _sdpa(q, K, V, scale), rtol=0, atol=1e-12)


def test_attention_length_one_is_v0():
    r = np.random.default_rng(1)
    q, K, V = r.normal(size=(4, 8)), r.normal(size=(1, 2, 8)), r.normal(size=(1, 2, 8))
    out = attention.decode_attention(q, K, V, 0.35)
    assert np.array_equal(out[:2], np.repeat(V[0, :1], 2, 0))
    assert np.array_equal(out[2:], np.repeat(V[0, 1:], 2, 0))


def test_attention_constant_keys_gives_mean():
    r = np.random.default_rng(2)
    L = 37
    q = r.normal(size=(2, 16))
    K = np.repeat(r.normal(size=(1, 1, 16)), L, 0)
    V = r.normal(size=(L, 1, 16))
    out = attention.decode_attention(q, K, V, 0.25)
    np.testing.assert_allclose(out, np.repeat(V.mean(0), 2, 0), atol=1e-14)


def test_attention_two_tokens_closed_form():
    """L = 2: out = v0 + sigmoid(s1 - s0) (v1 - v0)."""
    r = np.random.default_rng(3)
    q, K, V = r.normal(size=(1, 8)), r.normal(size=(2, 1, 8)), r.normal(size=(2, 1, 8))
    sc = 0.3
    s0, s1 = sc * K[0, 0] @ q[0], sc * K[1, 0] @ q[0]
    expect = V[0, 0] + (V[1, 0] - V[0, 0]) / (1 + math.exp(s0 - s1))
    np.testing.assert_allclose(attention.decode_attention(q, K, V, sc)[0], expect, atol=1e-14)


def test_attention_scale_and_sign():
    """A key aligned with q and a large scale selects its value row."""
    D = 8
    q = np.zeros((1, D)); q[0, 0] = 1.0
    K = np.zeros((3, 1, D)); K[1, 0, 0] = 1.0; K[2, 0, 0] = -1.0
    V = np.arange(3 * D, dtype=np.float64).reshape(3, 1, D)
    out = attention.decode_attention(q, K, V, 60.0)
    np.testing.assert_allclose(out[0], V[1, 0], atol=1e-20 + 1e-12)
    out0 = attention.decode_attention(q, K, V, 0.0)       # scale 0: uniform weights
    np.testing.assert_allclose(out0[0], V[:, 0].mean(0), atol=1e-14)


def test_paged_matches_contiguous_with_scrambled_tables():
    g = golden("p2_attention_small.json")
    r = np.random.default_rng(11)
    L, b, Hq, Hkv, D = g["length"], g["block_size"], g["q_heads"], g["kv_heads"], g["head_dim"]
    N = 16
    t = blocks.SeqTables(N, b, r.permutation(N))
    t.create(0)
    t.reserve(0, L)
    K = r.normal(size=(L, Hkv, D)).astype(np.float32)
    V = r.normal(size=(L, Hkv, D)).astype(np.float32)
    pk = cache_ops.new_pool(N, Hkv, b, D, torch.float32)
    pv = cache_ops.new_pool(N, Hkv, b, D, torch.float32)
    cache_ops.append(pk, pv, torch.tensor(K), torch.tensor(V),
                     [t.slot(0, p) for p in range(L)], b)
    q = r.normal(size=(Hq, D)).astype(np.float32)
    scale = 1 / math.sqrt(D)
    paged = attention.paged_decode(q, pk, pv, t.tables[0], L, b, scale)
    contiguous = _sdpa(q.astype(np.float64), K.astype(np.float64), V.astype(np.float64), scale)
    assert np.abs(paged - contiguous).max() <= g["atol"]
    assert np.abs(paged - contiguous).max() < 1e-12
    # the physical placement does not matter at all: a second, differently
    # scrambled pool gives the identical result
    t2 = blocks.SeqTables(N, b, r.permutation(N))
    t2.create(0)
    t2.reserve(0, L)
    pk2 = cache_ops.new_pool(N, Hkv, b, D, torch.float32)
    pv2 = cache_ops.new_pool(N, Hkv, b, D, torch.float32)
    cache_ops.append(pk2, pv2, torch.tensor(K), torch.tensor(V),
                     [t2.slot(0, p) for p in range(L)], b)
    assert t2.tables[0] != t.tables[0]
    assert np.array_equal(paged, attention.paged_decode(q, pk2, pv2, t2.tables[0], L, b, scale))


@pytest.mark.parametrize("L,b,P", [(1, 16, 512), (40, 16, 16), (1000, 16, 512), (1025, 32, 512),
                                   (513, 16, 64), (77, 8, 24)])
def test_split_merge_equals_definition(L, b, P):
    r = np.random.default_rng(L + b + P)
    Hq, Hkv, D = 8, 2, 16
    q, K, V = r.normal(size=(Hq, D)), r.normal(size=(L, Hkv, D)), r.normal(size=(L, Hkv, D))
    a = attention.decode_attention(q, K, V, 0.25)
    s = attention.decode_attention_split(q, K, V, 0.25, b, P)
    np.testing.assert_allclose(s, a, rtol=0, atol=1e-13)


def test_merge_with_empty_state_is_identity():
    st = (0.5, 2.0, np.array([1.0, -1.0]))
    empty = (-np.inf, 0.0, np.zeros(2))
    for m in (attention.merge(st, empty), attention.merge(empty, st)):
        assert m[0] == st[0] and m[1] == st[1] and np.array_equal(m[2], st[2])


def test_merge_closed_form():
    """Merging two one-token states equals the two-token softmax."""
    s0, s1 = 0.7, -1.3
    v0, v1 = np.array([1.0, 2.0]), np.array([-3.0, 0.5])
    m, l, O = attention.merge(attention.local_statistics(np.array([s0]), v0[None]),
                              attention.local_statistics(np.array([s1]), v1[None]))
    w1 = 1 / (1 + math.exp(s0 - s1))
    np.testing.assert_allclose(O / l, (1 - w1) * v0 + w1 * v1, atol=1e-15)
    assert m == s0
