"""pa_decode_append (each sequence's newest K/V row written, then decode) against
the oracle's append followed by its decode (needs a GPU).

"25. Paged attention and prefix caching", "The paged cache": a decode step
first writes the step's keys and values into the pool, then attends over the
history that now includes them.  The pools must end bit for bit as the
oracle's append leaves them and the outputs must match the oracle's decode of
those pools; the launch that fuses both (16-bit pools, tensor-core kernel) and
the two-launch path (fp32, CUDA-core kernel) are held to the same bar.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import blocks as oblocks
from oracle import cache_ops as ocache

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 1e-2}


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_66_gb300 import api as _api
    return _api


@pytest.fixture(params=["simt", "mma", "mma-h1"])
def kernel(request, api):
    """Run a decode test once per partition kernel: CUDA cores, tensor cores (KV heads per CTA
    chosen per launch: two for 16-bit pools), tensor cores with one KV head per CTA forced."""
    name = request.param
    api.pa_set_decode_kernel("simt" if name == "simt" else "mma")
    api.pa_set_decode_heads_per_cta(1 if name == "mma-h1" else 0)
    yield "simt" if name == "simt" else "mma"
    api.pa_set_decode_kernel("auto")
    api.pa_set_decode_heads_per_cta(0)


def _rand(shape, dtype, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def _setup(lengths, Hq, Hkv, D, b, dtype, gen):
    """Scrambled pool holding every position (the newest one with stale data)."""
    need = sum(-(-L // b) for L in lengths)
    N = need + 3
    t = oblocks.SeqTables(N, b, torch.randperm(N, generator=gen).tolist())
    for s, L in enumerate(lengths):
        t.create(s)
        t.reserve(s, L)
        t.advance(s, L)
    K = _rand((N, Hkv, b, D), dtype, gen)
    V = _rand((N, Hkv, b, D), dtype, gen)
    rows, lens = t.batch(range(len(lengths)))
    tables = torch.tensor(rows, dtype=torch.int32)
    slots = torch.tensor([t.tables[s][(L - 1) // b] * b + (L - 1) % b if L > 0 else -1
                          for s, L in enumerate(lengths)], dtype=torch.int64)
    B = len(lengths)
    q = _rand((B, Hq, D), dtype, gen)
    k_new = _rand((B, Hkv, D), dtype, gen)
    v_new = _rand((B, Hkv, D), dtype, gen)
    return K, V, tables, torch.tensor(lens, dtype=torch.int32), slots, q, k_new, v_new


def _run(api, q, k_new, v_new, slots, K, V, tables, lens, scale, part=0):
    B, Hq, D = q.shape
    n = api.pa_decode_workspace_size(B, Hq, D, tables.shape[1], K.shape[2], part)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda") if n else None
    Kd, Vd = K.cuda(), V.cuda()
    out = torch.full_like(q.cuda(), float("nan"))
    api.pa_decode_append(out, q.cuda(), k_new.cuda(), v_new.cuda(), slots.cuda(), Kd, Vd, tables.cuda(),
                         lens.cuda(), scale, partition_tokens=part, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu(), Kd.cpu(), Vd.cpu()


def _oracle(q, k_new, v_new, slots, K, V, tables, lens, b, scale):
    Kw, Vw = K.clone(), V.clone()
    ocache.append(Kw, Vw, k_new, v_new, slots, b)
    Kd, Vd = Kw.double().numpy(), Vw.double().numpy()
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(q.shape[0]):
        out[s] = oatt.paged_decode(q[s].double().numpy(), Kd, Vd, tables[s].tolist(), int(lens[s]), b, scale)
    return out, Kw, Vw


CASES = [
    # (Hq, Hkv, D, b, lengths, partition)
    (4, 2, 64, 16, [1, 7, 16, 17, 33], 0),
    (32, 8, 128, 16, [20, 511, 512, 513, 1000, 1537], 0),
    (32, 8, 128, 16, [20, 511, 512, 513, 1000], 64),       # the newest row in the 8th..16th partition
    (32, 4, 128, 32, [1, 32, 33, 700, 2049], 0),
    (12, 3, 128, 16, [100, 700, 1], 0),                      # odd Hkv: a CTA with one head
    (8, 1, 128, 64, [1, 65, 900], 0),                        # MQA, b = 64
    (16, 2, 256, 16, [1, 200, 900], 0),
    (32, 8, 128, 256, [1, 255, 256, 257, 1500], 0),
    (16, 4, 64, 16, [0, 300, 0, 1025], 0),                   # empty sequences (slot -1)
    (32, 8, 128, 48, [1, 48, 49, 700], 480),                 # three 16-token tiles per block
    (8, 2, 128, 240, [1, 240, 241, 1500], 480),              # fifteen tiles per block
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_decode_append_matches_oracle(api, kernel, dtype, case):
    Hq, Hkv, D, b, lengths, part = case
    if kernel == "mma" and dtype == torch.float32:
        pytest.skip("tensor-core kernel is for 16-bit pools")
    gen = torch.Generator().manual_seed(hash((Hq, Hkv, D, b, len(lengths), part, 5)) & 0xFFFF)
    K, V, tables, lens, slots, q, k_new, v_new = _setup(lengths, Hq, Hkv, D, b, dtype, gen)
    scale = 1 / math.sqrt(D)
    got, Kg, Vg = _run(api, q, k_new, v_new, slots, K, V, tables, lens, scale, part)
    want, Kw, Vw = _oracle(q, k_new, v_new, slots, K, V, tables, lens, b, scale)
    assert api.pa_get_device_error() == 0
    assert torch.equal(Kg, Kw) and torch.equal(Vg, Vw)
    err = np.abs(got.double().numpy() - want).max()
    assert err <= TOL[dtype], err


def test_decode_append_equals_append_then_decode(api):
    """The fused launch and the two launches give the same pools and the same
    outputs bit for bit (same kernel, same partitions, same arithmetic)."""
    gen = torch.Generator().manual_seed(21)
    K, V, tables, lens, slots, q, k_new, v_new = _setup([3, 512, 513, 2000, 777], 32, 8, 128, 16,
                                                        torch.float16, gen)
    scale = 128 ** -0.5
    got, Kg, Vg = _run(api, q, k_new, v_new, slots, K, V, tables, lens, scale)
    Kd, Vd = K.cuda(), V.cuda()
    api.pa_kv_append(k_new.cuda(), v_new.cuda(), Kd, Vd, slots.cuda())
    n = api.pa_decode_workspace_size(5, 32, 128, tables.shape[1], 16, 0)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda") if n else None
    out = torch.empty_like(q.cuda())
    api.pa_decode(out, q.cuda(), Kd, Vd, tables.cuda(), lens.cuda(), scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Kg, Kd.cpu()) and torch.equal(Vg, Vd.cpu())
    assert torch.equal(got, out.cpu())
    assert api.pa_get_device_error() == 0


def test_decode_append_negative_slot_writes_nothing(api):
    gen = torch.Generator().manual_seed(22)
    K, V, tables, lens, slots, q, k_new, v_new = _setup([40, 600], 8, 2, 64, 16, torch.bfloat16, gen)
    slots[1] = -1
    got, Kg, Vg = _run(api, q, k_new, v_new, slots, K, V, tables, lens, 0.125)
    want, Kw, Vw = _oracle(q, k_new, v_new, slots, K, V, tables, lens, 16, 0.125)
    assert torch.equal(Kg, Kw) and torch.equal(Vg, Vw)
    assert np.abs(got.double().numpy() - want).max() <= 1e-2
    assert api.pa_get_device_error() == 0


def test_decode_append_wrong_slot_is_flagged_and_skipped(api):
    """A slot that is not the table's slot of position L - 1 is not written and
    flags PA_DEVERR_SLOT; the other sequences are unaffected."""
    api.pa_set_decode_kernel("mma")
    try:
        gen = torch.Generator().manual_seed(23)
        K, V, tables, lens, slots, q, k_new, v_new = _setup([40, 600, 90], 8, 2, 64, 16, torch.float16, gen)
        bad = slots.clone()
        bad[1] = slots[1] - 1                        # the slot of position L - 2
        got, Kg, Vg = _run(api, q, k_new, v_new, bad, K, V, tables, lens, 0.125)
        assert api.pa_get_device_error() == 1        # PA_DEVERR_SLOT only
        keep = slots.clone()
        keep[1] = -1
        want, Kw, Vw = _oracle(q, k_new, v_new, keep, K, V, tables, lens, 16, 0.125)
        assert torch.equal(Kg, Kw) and torch.equal(Vg, Vw)
        assert np.abs(got.double().numpy() - want).max() <= 2e-3
    finally:
        api.pa_set_decode_kernel("auto")


def test_replay_fused_and_unfused_steps_agree(api):
    """Whole decode steps of the churn workload through pa_decode_append and
    through pa_kv_append + pa_decode: the same pools and outputs, bit for bit."""
    from paged_kv_cache_66_gb300.replay import Replay
    from workload import configs
    wl = configs.config2()
    a = Replay(wl, device="cuda", fused=True)
    u = Replay(wl, device="cuda", fused=False)
    assert a.fused and not u.fused
    a.run_setup()
    u.run_setup()
    for s in range(12):
        oa = a.run_step(a.device_step(a.plan_step(s)))
        ou = u.run_step(u.device_step(u.plan_step(s)))
        for x, y in zip(oa, ou):
            assert torch.equal(x, y)
    torch.cuda.synchronize()
    for li in range(len(a.layers)):
        assert torch.equal(a.k_pools[li], u.k_pools[li]) and torch.equal(a.v_pools[li], u.v_pools[li])
    assert api.pa_get_device_error() == 0
