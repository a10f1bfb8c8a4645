"""Decode through block tables built by the hash-chain prefix table (needs a GPU).

The shape of [P1] "Prefix caching"'s example: requests share a system prompt;
each attaches the cached blocks of its longest cached prefix, prefills
(appends K/V for) the rest, publishes its full blocks and then decodes one
token.  The K/V rows of a position are a function of the salt and the whole
token prefix up to that position (as in a model, where they depend on every
earlier token), so a reused block must hold exactly what the request would
have written itself.  Attention is checked against the oracle over each
request's own contiguous history.
"""
import hashlib
import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt

pytestmark = pytest.mark.gpu

HQ, HKV, D, B, N = 8, 2, 128, 16, 64


def _rows(salt, tokens):
    """fp16 K, V rows [Hkv, D] of the last position of ``tokens`` (input generator)."""
    seed = int.from_bytes(hashlib.sha256(salt + np.asarray(tokens, np.int64).tobytes()).digest()[:8], "little")
    r = np.random.default_rng(seed)
    return (r.standard_normal((2, HKV, D)).astype(np.float16))


def test_decode_through_hash_chain_prefix_tables():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_66_gb300 import api
    from paged_kv_cache_66_gb300.host import HostBlockManager, prefix_salt

    h = HostBlockManager(N, B)
    kp = torch.full((N, HKV, B, D), float("nan"), dtype=torch.float16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    system = list(range(1000, 1096))                                  # 96 tokens = 6 full blocks
    rev_a, rev_b = prefix_salt("rev-a"), prefix_salt("rev-b")
    requests = [(r, system + [r * 100 + i for i in range(8)], rev_a) for r in range(8)]
    requests += [(8, system + [5, 6], rev_b), (9, system + [7], rev_b)]          # another model revision
    requests += [(10, [1] + system[1:] + [9], rev_a)]                             # other first token
    expect_reused = [0] + [96] * 7 + [0, 96, 0]
    history = {}
    for (seq, prompt, salt), want in zip(requests, expect_reused):
        reused = h.hprefix_attach(seq, prompt, salt)
        assert reused == want
        n = len(prompt) - reused
        assert h.reserve(seq, n) == []                          # attached blocks are full
        slots = h.slots(seq, reused, n)
        kv = np.stack([_rows(salt, prompt[:p + 1]) for p in range(reused, len(prompt))])   # [n, 2, Hkv, D]
        api.pa_kv_append(torch.from_numpy(kv[:, 0]).cuda(), torch.from_numpy(kv[:, 1]).cuda(), kp, vp,
                         torch.from_numpy(slots).cuda())
        h.advance(seq, n)
        h.hprefix_remember(seq, prompt, salt)
        history[seq] = (list(prompt), salt)
    # one decode step for every request
    seqs = [r[0] for r in requests]
    new_slots, new_rows = [], []
    for seq in seqs:
        toks, salt = history[seq]
        toks.append(5000 + seq)
        assert h.reserve(seq, 1) == []
        new_slots.append(int(h.slots(seq, len(toks) - 1, 1)[0]))
        new_rows.append(_rows(salt, toks))
        h.advance(seq, 1)
    kv = np.stack(new_rows)
    api.pa_kv_append(torch.from_numpy(kv[:, 0]).cuda(), torch.from_numpy(kv[:, 1]).cuda(), kp, vp,
                     torch.tensor(new_slots, dtype=torch.int64, device="cuda"))
    tables, lens = h.batch(seqs)
    q = torch.from_numpy(np.random.default_rng(5).standard_normal((len(seqs), HQ, D)).astype(np.float16))
    out = torch.empty_like(q).cuda()
    n_ws = api.pa_decode_workspace_size(len(seqs), HQ, D, tables.shape[1], B, 64)
    ws = torch.empty(n_ws, dtype=torch.uint8, device="cuda") if n_ws else None
    api.pa_decode(out, q.cuda(), kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                  1 / math.sqrt(D), partition_tokens=64, workspace=ws)
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    # blocks in use: 6 shared system blocks per revision (rev-a twice: two first tokens) + private tails
    private = sum(-(-len(history[s][0]) // B) - (6 if e == 96 else 0) for s, e in zip(seqs, expect_reused))
    assert N - h.num_free == private
    got = out.cpu().double().numpy()
    for i, seq in enumerate(seqs):
        toks, salt = history[seq]
        rows = np.stack([_rows(salt, toks[:p + 1]) for p in range(len(toks))]).astype(np.float64)
        want = oatt.decode_attention(q[i].double().numpy(), rows[:, 0], rows[:, 1], 1 / math.sqrt(D))
        assert np.abs(got[i] - want).max() <= 2e-3
