"""Paged prefill on the GPU against the oracle (needs a GPU).

Pools hold random values; slots past each sequence's length hold NaN, so any
read of an unwritten slot shows.  The oracle computes each chunk row's causal
attention from the stored values in fp64; the kernel must match within the
tolerance of the storage dtype (f16 2e-3, bf16 1e-2, as for decode).
"""
import math

import numpy as np
import pytest
import torch

from oracle import blocks as oblocks
from oracle import prefill as oprefill

pytestmark = pytest.mark.gpu

TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
MANT = {torch.float16: 10, torch.bfloat16: 7}


def _check(got, want, V, dtype, visible):
    """Rows with >= 64 visible keys: the decode tolerance.  Every element: that
    tolerance plus the rounding bound of a few-key average, 2^-(m+1) (|o| +
    max|v|) -- P and the output are each rounded once to the dtype (m mantissa
    bits), which a short row does not average away."""
    err = np.abs(got - want)
    vmax = float(np.nanmax(np.abs(V)))
    bound = TOL[dtype] + 2.0 ** -(MANT[dtype] + 1) * (np.abs(want) + vmax)
    assert (err <= bound).all(), float((err - bound).max())
    long_rows = np.asarray(visible) >= 64
    if long_rows.any():
        assert err[long_rows].max() <= TOL[dtype]


def _visible(lengths, chunks):
    out = []
    for L, C in zip(lengths, chunks):
        out += [L - C + r + 1 for r in range(C)]
    return out


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_66_gb300 import api as _api
    return _api


def _setup(lengths, chunks, Hq, Hkv, D, b, dtype, seed, extra=5):
    gen = torch.Generator().manual_seed(seed)
    need = sum(-(-L // b) for L in lengths)
    N = need + extra
    t = oblocks.SeqTables(N, b, torch.randperm(N, generator=gen).tolist())
    for s, L in enumerate(lengths):
        t.create(s)
        t.reserve(s, L)
        t.advance(s, L)
    K = torch.randn((N, Hkv, b, D), generator=gen).to(dtype)
    V = torch.randn((N, Hkv, b, D), generator=gen).to(dtype)
    for s, L in enumerate(lengths):                       # unwritten tail slots: NaN
        if L % b:
            blk = t.tables[s][-1]
            K[blk, :, L % b:] = float("nan")
            V[blk, :, L % b:] = float("nan")
    rows, lens = t.batch(range(len(lengths)))
    qstart = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = torch.randn((int(qstart[-1]), Hq, D), generator=gen).to(dtype)
    return K, V, q, torch.tensor(rows, dtype=torch.int32), torch.tensor(lens, dtype=torch.int32), \
        torch.tensor(qstart, dtype=torch.int32)


def _run(api, K, V, q, tables, lens, qstart, scale, max_q=None):
    out = torch.full_like(q, float("nan")).cuda()
    api.pa_prefill(out, q.cuda(), K.cuda(), V.cuda(), tables.cuda(), lens.cuda(), qstart.cuda(), scale,
                   max_query_len=max_q)
    torch.cuda.synchronize()
    return out.cpu()


CASES = [
    # (Hq, Hkv, D, b, lengths, chunks)
    (32, 8, 128, 16, [100, 1, 64, 513], [100, 1, 20, 77]),
    (8, 8, 64, 16, [37, 300], [37, 129]),
    (16, 2, 256, 32, [70, 200], [70, 33]),
    (8, 4, 128, 32, [1000], [300]),
    (4, 1, 64, 16, [16, 17, 15], [16, 17, 15]),
    (32, 4, 128, 16, [47, 8], [47, 8]),
    (8, 1, 256, 16, [33], [2]),
    (8, 2, 128, 64, [300, 64], [150, 64]),             # b = 64
    (4, 4, 64, 256, [600], [600]),                      # b = 256, G = 1: 600 chunk rows over 3 CTAs
    (4, 4, 128, 16, [700], [700]),                      # G = 1, a whole 256-row CTA plus a ragged one
    (6, 3, 128, 16, [200, 90], [100, 90]),              # odd Hkv
    (16, 2, 128, 16, [1500, 777], [300, 777]),          # G = 8: many 128-key tiles, ragged ends
    (8, 2, 128, 256, [900], [400]),                     # b = 256 at D = 128
    (8, 2, 256, 16, [700, 150], [300, 150]),            # D = 256, G = 4: history + ragged chunk
    (4, 4, 256, 16, [300], [300]),                      # D = 256, G = 1: three 128-row CTAs
    (8, 4, 256, 32, [1000], [257]),                     # D = 256, G = 2, b = 32
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_prefill_matches_oracle(api, dtype, case):
    Hq, Hkv, D, b, lengths, chunks = case
    K, V, q, tables, lens, qstart = _setup(lengths, chunks, Hq, Hkv, D, b, dtype,
                                           seed=hash((Hq, D, b, len(lengths))) & 0xFFFF)
    scale = 1 / math.sqrt(D)
    got = _run(api, K, V, q, tables, lens, qstart, scale)
    assert api.pa_get_device_error() == 0
    want = oprefill.paged_prefill_batch(q.double().numpy(), K.double().numpy(), V.double().numpy(),
                                        tables.tolist(), lens.tolist(), qstart.tolist(), b, scale)
    assert torch.isfinite(got).all()
    _check(got.double().numpy(), want, V.double().numpy(), dtype, _visible(lengths, chunks))


def test_prefill_chunk_of_one_equals_decode(api):
    """A one-row chunk is decode at the sequence's last position."""
    Hq, Hkv, D, b = 32, 8, 128, 16
    lengths = [513, 40, 1]
    K, V, q, tables, lens, qstart = _setup(lengths, [1, 1, 1], Hq, Hkv, D, b, torch.float16, seed=9)
    got = _run(api, K, V, q, tables, lens, qstart, 0.088)
    out = torch.empty_like(q).cuda()
    n = api.pa_decode_workspace_size(3, Hq, D, tables.shape[1], b, 0)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda") if n else None
    api.pa_decode(out, q.cuda(), K.cuda(), V.cuda(), tables.cuda(), lens.cuda(), 0.088, workspace=ws)
    torch.cuda.synchronize()
    assert (got - out.cpu()).abs().max().item() <= 2e-3


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_inconsistent_chunk_is_flagged_and_skipped(api, D):
    Hq, Hkv, b = 8, 2, 16
    K, V, q, tables, lens, qstart = _setup([20, 30], [5, 6], Hq, Hkv, D, b, torch.float16, seed=11)
    lens[0] = 3                                           # chunk of 5 > length 3
    got = _run(api, K, V, q, tables, lens, qstart, 0.125)
    assert api.pa_get_device_error() == 4                 # PA_DEVERR_SEQLEN
    assert torch.isnan(got[:5]).all()                     # skipped rows stay unwritten
    want = oprefill.paged_prefill_batch(q[5:].double().numpy(), K.double().numpy(), V.double().numpy(),
                                        tables[1:].tolist(), lens[1:].tolist(), [0, 6], b, 0.125)
    assert np.abs(got[5:].double().numpy() - want).max() <= 2e-3


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_bad_table_entry_is_flagged(api, D):
    Hq, Hkv, b = 8, 2, 16
    K, V, q, tables, lens, qstart = _setup([40], [40], Hq, Hkv, D, b, torch.float16, seed=12)
    tables[0, 1] = K.shape[0] + 7
    _run(api, K, V, q, tables, lens, qstart, 0.125)
    assert api.pa_get_device_error() == 2                 # PA_DEVERR_TABLE


def test_prefill_d256_bad_entries_are_flagged_and_skipped(api):
    """The D = 256 tcgen05 kernel's error paths: an inconsistent chunk is skipped (rows stay
    unwritten) and flagged, the other sequence still matches the oracle; a table entry outside
    the pool is flagged."""
    Hq, Hkv, D, b = 8, 2, 256, 16
    K, V, q, tables, lens, qstart = _setup([20, 90], [5, 40], Hq, Hkv, D, b, torch.bfloat16, seed=41)
    lens[0] = 3                                           # chunk of 5 > length 3
    got = _run(api, K, V, q, tables, lens, qstart, 0.0625)
    assert api.pa_get_device_error() == 4                 # PA_DEVERR_SEQLEN
    assert torch.isnan(got[:5]).all()
    want = oprefill.paged_prefill_batch(q[5:].double().numpy(), K.double().numpy(), V.double().numpy(),
                                        tables[1:].tolist(), lens[1:].tolist(), [0, 40], b, 0.0625)
    _check(got[5:].double().numpy(), want, V.double().numpy(), torch.bfloat16, _visible([90], [40]))
    K, V, q, tables, lens, qstart = _setup([70], [70], Hq, Hkv, D, b, torch.bfloat16, seed=42)
    tables[0, 2] = K.shape[0] + 3
    _run(api, K, V, q, tables, lens, qstart, 0.0625)
    assert api.pa_get_device_error() == 2                 # PA_DEVERR_TABLE


def test_prefill_f32_unsupported(api):
    K, V, q, tables, lens, qstart = _setup([20], [20], 4, 2, 64, 16, torch.float32, seed=13)
    with pytest.raises(api.PagedKVError) as e:
        _run(api, K, V, q, tables, lens, qstart, 0.125)
    assert e.value.status == 2


@pytest.mark.parametrize("head_dim", [128, 64, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_bench_workload_sampled_rows(api, dtype, head_dim):
    """The benchmark's launch (8 chunks of 1024 over 3072 cached tokens, Llama-3-8B
    layer shape), inputs generated on the device as the benchmark does; sampled
    rows checked one by one against the oracle."""
    from oracle import attention as oatt
    from workload import configs as wcfg
    wl = wcfg.prefill_config(dtype=dtype, head_dim=head_dim)
    kp, vp, q = wcfg.prefill_inputs(wl, device="cuda")
    tables = torch.as_tensor(wl.tables(), device="cuda")
    lens = torch.full((wl.batch,), wl.length, dtype=torch.int32, device="cuda")
    qstart = torch.as_tensor(wl.qstart(), device="cuda")
    out = torch.empty_like(q)
    api.pa_prefill(out, q, kp, vp, tables, lens, qstart, wl.scale, max_query_len=wl.chunk)
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    K, V = kp.cpu(), vp.cpu()
    got, qc = out.cpu().double().numpy(), q.cpu().double().numpy()
    tol = TOL[wl.torch_dtype]
    for s, r in [(0, 0), (0, 511), (3, 1023), (7, 64), (7, 1023)]:
        pos = wl.history + r
        Kh = oatt.gather_history(K, wl.tables()[s], pos + 1, wl.b)
        Vh = oatt.gather_history(V, wl.tables()[s], pos + 1, wl.b)
        want = oprefill.prefill_attention(qc[s * wl.chunk + r][None], Kh, Vh, wl.scale)[0]
        assert np.abs(got[s * wl.chunk + r] - want).max() <= tol


@pytest.mark.parametrize("D", [64, 128, 256])
def test_prefill_many_units_per_cta_ragged(api, D):
    """More work units than SMs, so each persistent CTA walks many of them: chunks of 0 to 512
    rows (many units empty and skipped), one inconsistent sequence in the middle (flagged, its
    rows left unwritten), and sampled rows of every other sequence against the oracle."""
    from oracle import attention as oatt
    Hq, Hkv, b, dtype = 32, 8, 16, torch.bfloat16
    rng = np.random.default_rng(77 + D)
    chunks = [int(c) for c in rng.choice([0, 1, 37, 128, 256, 300, 512], size=24)]
    bad = 7
    chunks[5], chunks[11], chunks[bad] = 512, 0, 37
    lengths = [c + int(h) for c, h in zip(chunks, rng.integers(1, 300, size=24))]
    K, V, q, tables, lens, qstart = _setup(lengths, chunks, Hq, Hkv, D, b, dtype, seed=500 + D)
    lens[bad] = chunks[bad] - 1                           # a chunk longer than its sequence
    got = _run(api, K, V, q, tables, lens, qstart, 1 / math.sqrt(D), max_q=max(chunks))
    assert api.pa_get_device_error() == 4                 # PA_DEVERR_SEQLEN, and nothing else
    qs = qstart.tolist()
    assert torch.isnan(got[qs[bad]:qs[bad + 1]]).all()
    Kd, Vd, qd, gd = K.double(), V.double(), q.double().numpy(), got.double().numpy()
    for s in range(24):
        C = qs[s + 1] - qs[s]
        if s == bad or C == 0:
            continue
        L = int(lens[s])
        for r in sorted({0, C // 2, C - 1}):
            pos = L - C + r
            Kh = oatt.gather_history(Kd, tables[s].tolist(), pos + 1, b)
            Vh = oatt.gather_history(Vd, tables[s].tolist(), pos + 1, b)
            want = oprefill.prefill_attention(qd[qs[s] + r][None], Kh, Vh, 1 / math.sqrt(D))[0]
            _check(gd[qs[s] + r][None], want[None], Vh, dtype, [pos + 1])
