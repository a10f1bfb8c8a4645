"""Pins of the paged prefill oracle (CPU only).

Checked against: torch's scaled_dot_product_attention with is_causal in fp64
(a library routine; for a chunk that is the whole sequence the two causal
masks coincide), closed forms (a constant key gives the running mean of V;
the first position sees only v_0), the decode oracle for a chunk of one row,
chunk invariance (a chunk's rows equal the same rows of a longer chunk), and
placement invariance through scrambled block tables.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, prefill


def _sdpa_causal(q, K, V, scale):
    """q [L, Hq, D], K, V [L, Hkv, D] -> [L, Hq, D] via torch (fp64, GQA by repeat)."""
    Hq, Hkv = q.shape[1], K.shape[1]
    G = Hq // Hkv
    tq = torch.tensor(q).permute(1, 0, 2)
    tk = torch.tensor(K).permute(1, 0, 2).repeat_interleave(G, 0)
    tv = torch.tensor(V).permute(1, 0, 2).repeat_interleave(G, 0)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv,D,L", [(4, 2, 8, 1), (4, 2, 8, 37), (8, 1, 32, 16), (8, 8, 16, 33), (32, 8, 64, 70)])
def test_full_prefill_matches_library_causal_sdpa(Hq, Hkv, D, L):
    r = np.random.default_rng(L * 7 + D)
    q = r.normal(size=(L, Hq, D))
    K = r.normal(size=(L, Hkv, D))
    V = r.normal(size=(L, Hkv, D))
    got = prefill.prefill_attention(q, K, V, 1 / math.sqrt(D))
    np.testing.assert_allclose(got, _sdpa_causal(q, K, V, 1 / math.sqrt(D)), rtol=0, atol=1e-12)


def test_first_position_sees_only_v0_and_constant_keys_give_running_mean():
    r = np.random.default_rng(3)
    L, Hq, Hkv, D = 20, 4, 2, 8
    q = r.normal(size=(L, Hq, D))
    K = np.repeat(r.normal(size=(1, Hkv, D)), L, 0)          # every key equal
    V = r.normal(size=(L, Hkv, D))
    out = prefill.prefill_attention(q, K, V, 0.5)
    assert np.array_equal(out[0], np.repeat(V[0], 2, 0))     # exactly v_0 (weights 1)
    running = np.cumsum(V, 0) / np.arange(1, L + 1)[:, None, None]
    np.testing.assert_allclose(out, np.repeat(running, 2, 1), atol=1e-14)


def test_chunk_of_one_row_is_decode():
    r = np.random.default_rng(4)
    L, Hq, Hkv, D = 45, 8, 2, 16
    K, V = r.normal(size=(L, Hkv, D)), r.normal(size=(L, Hkv, D))
    q = r.normal(size=(1, Hq, D))
    got = prefill.prefill_attention(q, K, V, 0.25)[0]
    assert np.array_equal(got, attention.decode_attention(q[0], K, V, 0.25))


@pytest.mark.parametrize("C", [1, 5, 16, 30])
def test_chunk_rows_equal_rows_of_the_whole_prefill(C):
    r = np.random.default_rng(5 + C)
    L, Hq, Hkv, D = 30, 4, 1, 8
    K, V = r.normal(size=(L, Hkv, D)), r.normal(size=(L, Hkv, D))
    q = r.normal(size=(L, Hq, D))
    whole = prefill.prefill_attention(q, K, V, 0.3)
    part = prefill.prefill_attention(q[L - C:], K, V, 0.3)
    assert np.array_equal(part, whole[L - C:])


def test_paged_batch_equals_contiguous_under_scrambled_tables():
    r = np.random.default_rng(6)
    b, Hq, Hkv, D, N = 4, 4, 2, 8, 40
    lengths, chunks = [9, 1, 16, 23], [3, 1, 16, 7]
    K = r.normal(size=(N, Hkv, b, D))
    V = r.normal(size=(N, Hkv, b, D))
    perm = r.permutation(N).tolist()
    tables, at = [], 0
    for L in lengths:
        n = -(-L // b)
        tables.append(perm[at:at + n] + [0] * 3)
        at += n
    qstart = np.concatenate([[0], np.cumsum(chunks)])
    q = r.normal(size=(int(qstart[-1]), Hq, D))
    got = prefill.paged_prefill_batch(q, K, V, tables, lengths, qstart, b, 0.4)
    for s, L in enumerate(lengths):
        Kc = attention.gather_history(K, tables[s], L, b)
        Vc = attention.gather_history(V, tables[s], L, b)
        want = prefill.prefill_attention(q[qstart[s]:qstart[s + 1]], Kc, Vc, 0.4)
        assert np.array_equal(got[qstart[s]:qstart[s + 1]], want)
    # brute force for one row: position 8 of sequence 0 sees its 9 positions
    row = qstart[1] - 1
    Kc = np.stack([K[tables[0][p // b], :, p % b] for p in range(9)])
    Vc = np.stack([V[tables[0][p // b], :, p % b] for p in range(9)])
    for h in range(Hq):
        s = 0.4 * Kc[:, h // 2] @ q[row, h]
        w = np.exp(s - s.max())
        np.testing.assert_allclose(got[row, h], w @ Vc[:, h // 2] / w.sum(), atol=1e-13)


def test_chunk_longer_than_sequence_rejected():
    with pytest.raises(ValueError):
        prefill.prefill_attention(np.zeros((3, 2, 4)), np.zeros((2, 1, 4)), np.zeros((2, 1, 4)), 1.0)
