"""pa_decode_noalloc, the decode entry point for callers that cannot allocate
device memory (an application that owns all device memory through its own
allocator, a loop that must not allocate after start-up, an ABI consumer with
no allocator): its split-K scratch is a fixed array inside the library.

Called through the C ABI on two calls in a row with different inputs (the
shared array keeps the first call's contents).  Each result must equal, bit
for bit, pa_decode with caller-provided scratch -- the same kernels on the
same inputs -- and match the fp64 oracle within the fp16 decode tolerance.
Free device memory must not change across the second call: it allocates
nothing.  Runs alone in a fresh process as well as after the rest of the
suite.
"""
import ctypes as C
import math

import pytest
import torch

pytestmark = pytest.mark.gpu

F16 = 1


def _paged_inputs(lengths, Hq, Hkv, D, b, seed):
    g = torch.Generator().manual_seed(seed)
    need = sum(-(-L // b) for L in lengths)
    N = need + 5
    perm = torch.randperm(N, generator=g)
    width = max(-(-L // b) for L in lengths)
    tables = torch.zeros((len(lengths), width), dtype=torch.int32)
    k = 0
    for s, L in enumerate(lengths):
        nb = -(-L // b)
        tables[s, :nb] = perm[k:k + nb].to(torch.int32)
        k += nb
    Kp = torch.randn((N, Hkv, b, D), generator=g).to(torch.float16)
    Vp = torch.randn((N, Hkv, b, D), generator=g).to(torch.float16)
    q = torch.randn((len(lengths), Hq, D), generator=g).to(torch.float16)
    lens = torch.tensor(lengths, dtype=torch.int32)
    return [x.cuda() for x in (q, Kp, Vp, tables, lens)]


def _p(t):
    return C.c_void_p(t.data_ptr())


def test_noalloc_decode_matches_caller_scratch_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import numpy as np

    from oracle import attention as oatt
    from paged_kv_cache_66_gb300 import _lib, api
    lib = _lib.load()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [([3000, 700, 1, 4096], 32, 8, 128, 16, 11),     # 8 partitions of 512 tokens
             ([5000, 33, 2048], 16, 2, 256, 32, 12)]          # different shape, more partitions
    for call, (lengths, Hq, Hkv, D, b, seed) in enumerate(cases):
        q, Kp, Vp, tables, lens = _paged_inputs(lengths, Hq, Hkv, D, b, seed)
        B = len(lengths)
        scale = 1.0 / math.sqrt(D)
        assert api.pa_decode_workspace_size(B, Hq, D, tables.shape[1], b, 0) > 0   # scratch is in use
        ref = torch.empty_like(q)
        api.pa_decode(ref, q, Kp, Vp, tables, lens, scale,
                      workspace=torch.empty(api.pa_decode_workspace_size(B, Hq, D, tables.shape[1], b, 0),
                                            dtype=torch.uint8, device="cuda"))
        out = torch.full_like(q, float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = lib.pa_decode_noalloc(_p(out), _p(q), _p(Kp), _p(Vp), Kp.shape[0], _p(tables), tables.shape[1],
                                   _p(lens), B, Hq, Hkv, D, b, scale, 0, F16, stream)
        assert st == 0, lib.pa_status_string(st)
        torch.cuda.synchronize()
        if call == 1:
            # the array was set up by the first call; this one must take no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.equal(out, ref)
        Kc, Vc, qc, tc = Kp.cpu(), Vp.cpu(), q.cpu().double().numpy(), tables.cpu().tolist()
        for s_, L in enumerate(lengths):
            want = oatt.paged_decode(qc[s_], Kc, Vc, tc[s_], L, b, scale)
            err = float(np.abs(out[s_].cpu().double().numpy() - want).max())
            assert err <= 2e-3, (call, s_, err)
    assert api.pa_get_device_error() == 0


def test_noalloc_rejects_batches_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_66_gb300 import _lib
    lib = _lib.load()
    # 64 x 32 heads x 64 partitions x (128 + 2) floats = 68 MB > 16 MiB: refused before any launch
    null = C.c_void_p(0)
    st = lib.pa_decode_noalloc(null, null, null, null, 20000, null, 2048, null, 64, 32, 8, 128, 16, 0.088, 0, F16,
                               null)
    assert lib.pa_status_string(st).decode() == "PA_ERR_INVALID"
