"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch each one.  This shows the pins constrain the oracle, not just agree with it."""
import numpy as np
import pytest

from oracle import attention, blocks
from tests import test_oracle_pins as pins


def _attention_gqa_modulo(q, K, V, scale):
    q, K, V = (np.asarray(x, dtype=np.float64) for x in (q, K, V))
    Hq, D = q.shape
    Hkv = K.shape[1]
    out = np.zeros((Hq, D))
    for h in range(Hq):
        g = h % Hkv                                   # wrong grouping
        s = scale * (K[:, g, :] @ q[h])
        p = np.exp(s - s.max())
        out[h] = (p @ V[:, g, :]) / p.sum()
    return out


def _attention_no_scale(q, K, V, scale):
    return _ORIG_ATT(q, K, V, 1.0)


def _attention_transposed_kv(q, K, V, scale):
    return _ORIG_ATT(q, V, K, scale)


_ORIG_ATT = attention.decode_attention


@pytest.mark.parametrize("bad", [_attention_gqa_modulo, _attention_no_scale,
                                 _attention_transposed_kv])
def test_attention_mistakes_are_caught(monkeypatch, bad):
    monkeypatch.setattr(attention, "decode_attention", bad)
    with pytest.raises(AssertionError):
        pins.test_attention_matches_library_sdpa(8, 2, 32, 17)


def test_merge_without_rescale_is_caught(monkeypatch):
    def bad_merge(a, b):
        (ma, la, Oa), (mb, lb, Ob) = a, b
        if la == 0:
            return b
        if lb == 0:
            return a
        return max(ma, mb), la + lb, Oa + Ob           # dropped exp(m - m') factors
    monkeypatch.setattr(attention, "merge", bad_merge)
    with pytest.raises(AssertionError):
        pins.test_split_merge_equals_definition(1000, 16, 512)


def test_swapped_slot_encoding_is_caught(monkeypatch):
    def bad_slot(self, seq, pos):
        table = self.tables[seq]
        return (pos % self.block_size) * self.block_size + table[pos // self.block_size]
    monkeypatch.setattr(blocks.SeqTables, "slot", bad_slot)
    with pytest.raises((AssertionError, IndexError)):
        pins.test_append_gather_roundtrip_scrambled()


def test_missing_copy_on_write_is_caught(monkeypatch):
    def reserve_no_cow(self, seq, new_tokens):
        table = self.tables[seq]
        need = self.blocks_needed(self.lengths[seq] + int(new_tokens))
        while len(table) < need:
            table.append(self.allocator.allocate())
        return []
    monkeypatch.setattr(blocks.SeqTables, "reserve", reserve_no_cow)
    with pytest.raises(AssertionError):
        pins.test_cow_keeps_parent_history()
    with pytest.raises(AssertionError):
        pins.test_fork_cow_p1_numbers()


def test_lifo_free_list_is_caught(monkeypatch):
    def lifo_allocate(self):
        if not self.free:
            raise MemoryError("KV block pool exhausted")
        block = self.free.pop()
        self.refs[block] = 1
        return block
    monkeypatch.setattr(blocks.BlockAllocator, "allocate", lifo_allocate)
    with pytest.raises(AssertionError):
        pins.test_allocator_fifo_and_refcounts()


def test_chain_without_parent_key_is_caught(monkeypatch):
    """A key of the block's own tokens only lets equal text under another history match."""
    from oracle import prefix_hash as ph
    from tests import test_oracle_prefix_hash as hp
    orig = ph.next_key
    monkeypatch.setattr(ph, "next_key", lambda parent, toks: orig(b"", toks))
    with pytest.raises(AssertionError):
        hp.test_same_block_text_under_different_history_differs()
    with pytest.raises(AssertionError):
        hp.test_hash_table_equals_tuple_table_on_traces(0)


def test_chain_without_salt_is_caught(monkeypatch):
    from oracle import prefix_hash as ph
    from tests import test_oracle_prefix_hash as hp
    orig = ph.root_key
    monkeypatch.setattr(ph, "root_key", lambda salt=b"": orig(b""))
    with pytest.raises(AssertionError):
        hp.test_salt_separates_every_key()
    with pytest.raises(AssertionError):
        hp.test_hash_table_equals_tuple_table_on_traces(0)


def _prefill_off_by_one(q, K, V, scale):
    """Causal bound p < i instead of p <= i (the first row then sees nothing)."""
    q = np.asarray(q, dtype=np.float64)
    C, L = q.shape[0], K.shape[0]
    out = np.zeros(q.shape)
    for r in range(C):
        out[r] = attention.decode_attention(q[r], K[:L - C + r], V[:L - C + r], scale)
    return out


def _prefill_no_mask(q, K, V, scale):
    q = np.asarray(q, dtype=np.float64)
    return np.stack([attention.decode_attention(q[r], K, V, scale) for r in range(q.shape[0])])


def _prefill_chunk_at_start(q, K, V, scale):
    """Chunk rows placed at positions 0 .. C-1 instead of the last C positions."""
    q = np.asarray(q, dtype=np.float64)
    return np.stack([attention.decode_attention(q[r], K[:r + 1], V[:r + 1], scale) for r in range(q.shape[0])])


@pytest.mark.parametrize("bad", [_prefill_off_by_one, _prefill_no_mask, _prefill_chunk_at_start])
def test_prefill_mistakes_are_caught(monkeypatch, bad):
    from oracle import prefill
    from tests import test_oracle_prefill as pp
    monkeypatch.setattr(prefill, "prefill_attention", bad)
    caught = 0
    for test in (lambda: pp.test_full_prefill_matches_library_causal_sdpa(4, 2, 8, 37),
                 pp.test_first_position_sees_only_v0_and_constant_keys_give_running_mean,
                 pp.test_chunk_of_one_row_is_decode,
                 lambda: pp.test_chunk_rows_equal_rows_of_the_whole_prefill(5)):
        try:
            test()
        except AssertionError:
            caught += 1
    assert caught >= 1


def test_tree_eviction_of_inner_nodes_is_caught(monkeypatch):
    """A prefix tree that drops any idle node (not only leaves) strands the longer prefixes
    below it: the hand-worked divergence case and the trace invariants catch it."""
    from oracle import prefix_tree as pt
    from tests import test_oracle_prefix_tree as tree_pins

    def evict_any(self, blocks_wanted):
        alloc = self.tables.allocator
        while alloc.num_free < int(blocks_wanted):
            idle = [n for n in self.nodes() if alloc.refs[n.block] == 1]
            if not idle:
                return
            victim = min(idle, key=lambda n: n.used)
            del victim.parent.children[victim.label]
            alloc.release(victim.block)

    monkeypatch.setattr(pt.BlockPrefixTree, "evict", evict_any)
    with pytest.raises(AssertionError):
        tree_pins.test_eviction_takes_leaves_where_the_flat_table_strands_a_prefix()
    with pytest.raises(AssertionError):
        tree_pins.test_tree_invariants_hold_on_traces_with_eviction(0)


def test_tree_attach_without_prefill_margin_is_caught(monkeypatch):
    """Reusing every full block of the prompt (no token left to prefill) is caught."""
    from oracle import prefix_tree as pt
    from tests import test_oracle_prefix_tree as tree_pins
    orig = pt.BlockPrefixTree.attach

    def attach_all(self, seq, prompt):
        return orig(self, seq, list(prompt) + [None])    # one phantom token: the last block counts

    monkeypatch.setattr(pt.BlockPrefixTree, "attach", attach_all)
    with pytest.raises(AssertionError):
        tree_pins.test_at_least_one_prompt_token_is_left_to_prefill()
