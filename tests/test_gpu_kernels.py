"""GPU parity of each kernel against the oracle, through the C ABI (needs a GPU).

Bit-exact for the byte-moving kernels (KV append, copy-on-write) over the
whole pool; within the attention tolerance of the dtype for decode
(fp32 1e-5, fp16 2e-3, bf16 1e-2 max-abs against the fp64 oracle).
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
DTYPES = [torch.float32, torch.float16, torch.bfloat16]


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


# ------------------------------------------------------------------ KV append

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,b,Hkv", [(64, 16, 2), (128, 16, 8), (256, 32, 4), (128, 32, 1)])
def test_kv_append_bit_exact(api, dtype, D, b, Hkv):
    g = torch.Generator().manual_seed(D * 7 + b)
    N = 37
    T = 131                                           # ragged: not a multiple of anything
    slots = torch.randperm(N * b, generator=g)[:T].to(torch.int64)
    slots[5] = -1                                     # padding rows are skipped
    slots[77] = -3
    k = _rand((T, Hkv, D), dtype, g)
    v = _rand((T, Hkv, D), dtype, g)
    kp_ref = _rand((N, Hkv, b, D), dtype, g)          # pre-existing contents must survive
    vp_ref = _rand((N, Hkv, b, D), dtype, g)
    kp, vp = kp_ref.cuda(), vp_ref.cuda()
    api.pa_kv_append(k.cuda(), v.cuda(), kp, vp, slots.cuda())
    ocache.append(kp_ref, vp_ref, k, v, slots.tolist(), b)
    torch.cuda.synchronize()
    assert torch.equal(kp.cpu(), kp_ref) and torch.equal(vp.cpu(), vp_ref)
    assert api.pa_get_device_error() == 0


def test_kv_append_empty_and_bad_slot(api):
    kp = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device="cuda")
    vp = torch.zeros_like(kp)
    k = torch.ones((0, 2, 64), dtype=torch.float16, device="cuda")
    api.pa_kv_append(k, k, kp, vp, torch.zeros(0, dtype=torch.int64, device="cuda"))
    k = torch.ones((2, 2, 64), dtype=torch.float16, device="cuda")
    api.pa_kv_append(k, k, kp, vp, torch.tensor([3, 4 * 16], dtype=torch.int64, device="cuda"))
    code = api.pa_get_device_error()
    assert code & 1                                  # PA_DEVERR_SLOT
    assert kp.float().sum().item() == 2 * 64         # the in-range row landed, the other was skipped
    assert api.pa_get_device_error() == 0            # cleared


# ------------------------------------------------------------------ copy-on-write

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_copy_blocks_bit_exact(api, dtype):
    g = torch.Generator().manual_seed(3)
    N, Hkv, b, D, layers = 64, 8, 16, 128, 3
    K = [_rand((N, Hkv, b, D), dtype, g) for _ in range(layers)]
    V = [_rand((N, Hkv, b, D), dtype, g) for _ in range(layers)]
    perm = torch.randperm(N, generator=g)
    pairs = torch.stack([perm[:9], perm[9:18]], 1).to(torch.int64)   # disjoint src / dst
    Kd, Vd = [x.cuda() for x in K], [x.cuda() for x in V]
    api.pa_copy_blocks(Kd, Vd, pairs.cuda())
    ocache.copy_blocks(K, V, pairs.tolist())
    torch.cuda.synchronize()
    for a, b_ in zip(Kd + Vd, K + V):
        assert torch.equal(a.cpu(), b_)
    assert api.pa_get_device_error() == 0


def test_copy_blocks_many_layers_and_bad_pair(api):
    N, layers = 8, 70                                  # more layers than one launch takes
    K = [torch.full((N, 1, 16, 64), float(i), dtype=torch.float16, device="cuda") for i in range(layers)]
    V = [x.clone() for x in K]
    for x in K:
        x[2].fill_(-1.0)
    api.pa_copy_blocks(K, V, torch.tensor([[2, 5], [1, 99]], dtype=torch.int64, device="cuda"))
    assert api.pa_get_device_error() & 8               # PA_DEVERR_PAIR for (1, 99)
    for i, x in enumerate(K):
        assert torch.all(x[5] == -1.0) and torch.all(x[1] == float(i))


# ------------------------------------------------------------------ decode

def _setup_paged(lengths, Hkv, D, b, dtype, gen, N=None, extra=3):
    """Scrambled pool: each sequence's blocks drawn from a random permutation."""
    need = sum(-(-L // b) for L in lengths)
    N = N or need + extra
    order = torch.randperm(N, generator=gen).tolist()
    t = oblocks.SeqTables(N, b, order)
    for s, L in enumerate(lengths):
        t.create(s)
        t.reserve(s, L)
        t.advance(s, L)
    K = _rand((N, Hkv, b, D), dtype, gen)
    V = _rand((N, Hkv, b, D), dtype, gen)
    rows, lens = t.batch(range(len(lengths)))
    return t, K, V, torch.tensor(rows, dtype=torch.int32), torch.tensor(lens, dtype=torch.int32)


def _run_decode(api, q, K, V, tables, lens, scale, part=0):
    B, Hq, D = q.shape
    ws_n = api.pa_decode_workspace_size(B, Hq, D, tables.shape[1], K.shape[2], part)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda") if ws_n else None
    out = torch.full_like(q.cuda(), float("nan"))
    api.pa_decode(out, q.cuda(), K.cuda(), V.cuda(), tables.cuda(), lens.cuda(), scale, partition_tokens=part,
                  workspace=ws)
    torch.cuda.synchronize()
    return out.cpu()


def _oracle_decode(q, K, V, tables, lens, b, scale):
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(q.shape[0]):
        out[s] = oatt.paged_decode(q[s].double().numpy(), K, V, tables[s].tolist(), int(lens[s]), b, scale)
    return out


CASES = [
    # (Hq, Hkv, D, b, lengths, partition)
    (4, 2, 64, 16, [1, 7, 15, 16, 17, 33, 34], 0),
    (32, 8, 128, 16, [20, 511, 512, 513, 1000, 1537], 0),
    (32, 8, 128, 16, [20, 511, 512, 513, 1000, 1537], 64),
    (32, 4, 128, 32, [1, 31, 32, 33, 700, 2049], 0),
    (32, 32, 64, 16, [3, 300, 1100], 0),
    (16, 2, 256, 16, [1, 200, 900], 0),
    (16, 2, 256, 32, [64, 513], 256),
    (8, 4, 128, 16, [16 * 37 + 5, 8], 0),
    (12, 3, 128, 16, [100, 700, 1], 0),                 # odd Hkv: the last CTA of a head pair has one head
    (8, 1, 128, 64, [1, 65, 900], 0),                   # MQA, b = 64
    (32, 8, 128, 256, [1, 255, 256, 257, 1500], 0),     # b = 256: one block per half partition
    (16, 4, 64, 128, [300, 1025], 0),
    # blocks of 3, 5, 6 and 15 tiles of 16 tokens: a tile finds its table entry by division
    (32, 8, 128, 48, [1, 47, 48, 49, 700, 1441], 480),
    (16, 4, 64, 80, [1, 79, 81, 1000], 400),
    (16, 2, 256, 96, [95, 97, 800], 480),
    (8, 2, 128, 240, [1, 239, 241, 1500], 480),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("case", CASES)
def test_decode_matches_oracle(api, kernel, dtype, case):
    Hq, Hkv, D, b, lengths, part = case
    if kernel == "mma" and dtype == torch.float32:
        pytest.skip("tensor-core kernel is for 16-bit pools (covered by the unsupported test)")
    gen = torch.Generator().manual_seed(hash((Hq, Hkv, D, b, len(lengths), part)) & 0xFFFF)
    t, K, V, tables, lens = _setup_paged(lengths, Hkv, D, b, dtype, gen)
    q = _rand((len(lengths), Hq, D), dtype, gen)
    scale = 1 / math.sqrt(D)
    got = _run_decode(api, q, K, V, tables, lens, scale, part).double().numpy()
    want = _oracle_decode(q, K, V, tables, lens, b, scale)
    err = np.abs(got - want).max()
    assert err <= TOL[dtype], err
    assert api.pa_get_device_error() == 0


def test_mma_kernel_rejects_fp32(api):
    gen = torch.Generator().manual_seed(9)
    t, K, V, tables, lens = _setup_paged([5], 2, 64, 16, torch.float32, gen)
    q = _rand((1, 4, 64), torch.float32, gen)
    api.pa_set_decode_kernel("mma")
    try:
        with pytest.raises(api.PagedKVError) as e:
            _run_decode(api, q, K, V, tables, lens, 0.125)
        assert e.value.status == 2                      # PA_ERR_UNSUPPORTED
    finally:
        api.pa_set_decode_kernel("auto")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_simt_and_mma_kernels_agree(api, dtype):
    gen = torch.Generator().manual_seed(10)
    lengths = [1, 17, 700, 2500]
    t, K, V, tables, lens = _setup_paged(lengths, 8, 128, 16, dtype, gen)
    q = _rand((4, 32, 128), dtype, gen)
    outs = {}
    for k in ("simt", "mma"):
        api.pa_set_decode_kernel(k)
        outs[k] = _run_decode(api, q, K, V, tables, lens, 0.088).double()
    api.pa_set_decode_kernel("auto")
    assert (outs["simt"] - outs["mma"]).abs().max().item() <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_heads_per_cta_does_not_change_results(api, dtype):
    """One or two KV heads per CTA of the tensor-core kernel: bit-identical outputs (odd Hkv:
    the last CTA of a pair has one head)."""
    gen = torch.Generator().manual_seed(31)
    t, K, V, tables, lens = _setup_paged([1, 300, 513, 1500, 47], 3, 128, 16, dtype, gen)
    q = _rand((5, 12, 128), dtype, gen)
    outs = {}
    try:
        api.pa_set_decode_kernel("mma")
        for h in (1, 2, 0):
            api.pa_set_decode_heads_per_cta(h)
            outs[h] = _run_decode(api, q, K, V, tables, lens, 128 ** -0.5)
    finally:
        api.pa_set_decode_kernel("auto")
        api.pa_set_decode_heads_per_cta(0)
    assert torch.equal(outs[1], outs[2]) and torch.equal(outs[1], outs[0])
    assert api.pa_get_device_error() == 0


@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_length_one_is_v0_exactly(api, kernel, dtype):
    if kernel == "mma" and dtype == torch.float32:
        pytest.skip("tensor-core kernel is for 16-bit pools")
    gen = torch.Generator().manual_seed(1)
    t, K, V, tables, lens = _setup_paged([1, 1, 1], 2, 128, 16, dtype, gen)
    q = _rand((3, 8, 128), dtype, gen)
    got = _run_decode(api, q, K, V, tables, lens, 0.09)
    for s in range(3):
        blk = int(tables[s, 0])
        for h in range(8):
            assert torch.equal(got[s, h], V[blk, h // 4, 0])


def test_decode_zero_length_writes_zeros(api, kernel):
    gen = torch.Generator().manual_seed(2)
    t, K, V, tables, lens = _setup_paged([5, 40], 2, 64, 16, torch.float16, gen)
    lens[0] = 0
    q = _rand((2, 4, 64), torch.float16, gen)
    got = _run_decode(api, q, K, V, tables, lens, 0.125)
    assert torch.all(got[0] == 0)
    want = _oracle_decode(q[1:], K, V, tables[1:], lens[1:], 16, 0.125)
    assert np.abs(got[1:].double().numpy() - want).max() <= 2e-3


def test_decode_partition_size_does_not_matter(api, kernel):
    gen = torch.Generator().manual_seed(4)
    lengths = [3000, 129, 4096, 1]
    t, K, V, tables, lens = _setup_paged(lengths, 8, 128, 16, torch.float16, gen)
    q = _rand((4, 32, 128), torch.float16, gen)
    outs = [_run_decode(api, q, K, V, tables, lens, 0.088, part).double() for part in (0, 64, 512, 4096, 8192)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2e-3


def test_decode_physical_placement_is_invisible(api, kernel):
    """Same logical history at two different physical placements: identical bits."""
    gen = torch.Generator().manual_seed(5)
    lengths = [777, 40]
    t, K, V, tables, lens = _setup_paged(lengths, 8, 128, 16, torch.bfloat16, gen, N=120)
    perm = torch.randperm(120, generator=gen)
    K2, V2 = torch.empty_like(K), torch.empty_like(V)
    K2[perm], V2[perm] = K, V                      # block i moves to perm[i]
    tables2 = perm[tables.long()].to(torch.int32)
    q = _rand((2, 32, 128), torch.bfloat16, gen)
    a = _run_decode(api, q, K, V, tables, lens, 0.088)
    c = _run_decode(api, q, K2, V2, tables2, lens, 0.088)
    assert torch.equal(a, c)


def test_decode_unwritten_slots_are_masked(api, kernel):
    """NaN garbage past the length in the tail block must not leak into the output."""
    gen = torch.Generator().manual_seed(6)
    t, K, V, tables, lens = _setup_paged([21], 2, 64, 16, torch.float16, gen)
    blk = int(tables[0, 1])
    K[blk, :, 5:] = float("nan")
    V[blk, :, 5:] = float("inf")
    q = _rand((1, 4, 64), torch.float16, gen)
    got = _run_decode(api, q, K, V, tables, lens, 0.125)
    want = _oracle_decode(q, K, V, tables, lens, 16, 0.125)
    assert np.isfinite(got.double().numpy()).all()
    assert np.abs(got.double().numpy() - want).max() <= 2e-3


def test_decode_bad_table_entry_is_flagged_not_faulted(api, kernel):
    gen = torch.Generator().manual_seed(7)
    t, K, V, tables, lens = _setup_paged([40, 40], 2, 64, 16, torch.float16, gen)
    tables[1, 1] = 10_000                           # outside the pool
    q = _rand((2, 4, 64), torch.float16, gen)
    got = _run_decode(api, q, K, V, tables, lens, 0.125)
    assert api.pa_get_device_error() & 2             # PA_DEVERR_TABLE
    want = _oracle_decode(q[:1], K, V, tables[:1], lens[:1], 16, 0.125)
    assert np.abs(got[:1].double().numpy() - want).max() <= 2e-3
    assert torch.isfinite(got[1]).all()
    lens[0] = 10_000                                 # above the table's capacity
    _run_decode(api, q, K, V, tables, lens, 0.125)
    assert api.pa_get_device_error() & 4             # PA_DEVERR_SEQLEN


def test_bounded_wait_gives_up_and_reports(api):
    """A wait that nothing satisfies ends after its limit with a timeout status;
    the context stays usable (a decode right after still matches the oracle)."""
    from paged_kv_cache_66_gb300 import _lib
    lib = _lib.load()
    import ctypes as C
    assert api.pa_get_device_error() == 0
    st = lib.pa_selftest_wait_timeout(2000, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    code = api.pa_get_device_error()
    assert code == 16                                   # PA_DEVERR_TIMEOUT only
    gen = torch.Generator().manual_seed(12)
    t, K, V, tables, lens = _setup_paged([600, 3], 2, 64, 16, torch.float16, gen)
    q = _rand((2, 4, 64), torch.float16, gen)
    got = _run_decode(api, q, K, V, tables, lens, 0.125)
    want = _oracle_decode(q, K, V, tables, lens, 16, 0.125)
    assert np.abs(got.double().numpy() - want).max() <= 2e-3
    assert api.pa_get_device_error() == 0
