"""FP8 (E4M3) KV cache on the GPU against the oracle (needs a GPU).

Append: the pool bytes must equal the oracle's quantiser (E4M3 written out
from its definition) bit for bit.  Decode: the attention over the dequantised
history (codes x per-head scale, fp64) must match within the tolerance of the
query dtype (f16 2e-3, bf16 1e-2), as for 16-bit pools.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import blocks as oblocks
from oracle import quant

pytestmark = pytest.mark.gpu

TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_66_gb300 import api as _api
    return _api


def _scales(Hkv, gen):
    return (torch.rand(Hkv, generator=gen) * 0.05 + 0.01).to(torch.float32)


@pytest.mark.parametrize("in_dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D,b,Hkv", [(128, 16, 8), (256, 32, 2), (64, 16, 4)])
def test_kv_append_fp8_bit_exact(api, in_dtype, D, b, Hkv):
    g = torch.Generator().manual_seed(D + b + Hkv)
    N, T = 29, 101
    slots = torch.randperm(N * b, generator=g)[:T].to(torch.int64)
    slots[7] = -1
    k = (torch.randn((T, Hkv, D), generator=g) * 3).to(in_dtype)
    v = (torch.randn((T, Hkv, D), generator=g) * 3).to(in_dtype)
    k[3, 0, :4] = torch.tensor([1e6, -1e6, 0.0, -0.0]).to(in_dtype)      # saturation and signed zeros
    ks, vs = _scales(Hkv, g), _scales(Hkv, g)
    kp0 = torch.randint(0, 256, (N, Hkv, b, D), generator=g, dtype=torch.uint8)
    vp0 = torch.randint(0, 256, (N, Hkv, b, D), generator=g, dtype=torch.uint8)
    kp, vp = kp0.cuda(), vp0.cuda()
    api.pa_kv_append_fp8(k.cuda(), v.cuda(), kp, vp, ks.cuda(), vs.cuda(), slots.cuda())
    torch.cuda.synchronize()
    want_k, want_v = kp0.numpy().copy(), vp0.numpy().copy()
    kq = quant.quantize_rows(k.float().numpy(), ks.numpy())
    vq = quant.quantize_rows(v.float().numpy(), vs.numpy())
    for t, sl in enumerate(slots.tolist()):
        if sl >= 0:
            want_k[sl // b, :, sl % b, :] = kq[t]
            want_v[sl // b, :, sl % b, :] = vq[t]
    assert np.array_equal(kp.cpu().numpy(), want_k)
    assert np.array_equal(vp.cpu().numpy(), want_v)
    assert api.pa_get_device_error() == 0


def _fp8_setup(lengths, Hkv, D, b, gen, extra=3):
    need = sum(-(-L // b) for L in lengths)
    N = need + extra
    t = oblocks.SeqTables(N, b, torch.randperm(N, generator=gen).tolist())
    for s, L in enumerate(lengths):
        t.create(s)
        t.reserve(s, L)
        t.advance(s, L)
    ks, vs = _scales(Hkv, gen), _scales(Hkv, gen)
    Kx = torch.randn((N, Hkv, b, D), generator=gen)
    Vx = torch.randn((N, Hkv, b, D), generator=gen)
    Kc = quant.quantize_rows(Kx.permute(0, 2, 1, 3).reshape(-1, Hkv, D).numpy(), ks.numpy())
    Vc = quant.quantize_rows(Vx.permute(0, 2, 1, 3).reshape(-1, Hkv, D).numpy(), vs.numpy())
    Kc = torch.tensor(Kc).reshape(N, b, Hkv, D).permute(0, 2, 1, 3).contiguous()
    Vc = torch.tensor(Vc).reshape(N, b, Hkv, D).permute(0, 2, 1, 3).contiguous()
    rows, lens = t.batch(range(len(lengths)))
    return Kc, Vc, ks, vs, torch.tensor(rows, dtype=torch.int32), torch.tensor(lens, dtype=torch.int32)


def _decode(api, q, Kc, Vc, ks, vs, tables, lens, scale, part=0):
    B, Hq, D = q.shape
    n = api.pa_decode_workspace_size(B, Hq, D, tables.shape[1], Kc.shape[2], part)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda") if n else None
    out = torch.full_like(q.cuda(), float("nan"))
    api.pa_decode_fp8(out, q.cuda(), Kc.cuda(), Vc.cuda(), ks.cuda(), vs.cuda(), tables.cuda(), lens.cuda(), scale,
                      partition_tokens=part, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu()


def _oracle(q, Kc, Vc, ks, vs, tables, lens, b, scale):
    K = quant.dequantize(Kc.numpy(), ks.numpy(), head_axis=1)
    V = quant.dequantize(Vc.numpy(), vs.numpy(), head_axis=1)
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(q.shape[0]):
        out[s] = oatt.paged_decode(q[s].double().numpy(), K, V, tables[s].tolist(), int(lens[s]), b, scale)
    return out


FP8_CASES = [
    # (Hq, Hkv, D, b, lengths, partition)
    (32, 8, 128, 16, [1, 15, 16, 17, 511, 512, 513, 1300], 0),
    (32, 8, 128, 16, [700, 3], 64),
    (8, 8, 128, 32, [33, 1000], 0),
    (16, 8, 128, 16, [250, 40], 0),
    (16, 2, 256, 16, [1, 200, 900], 0),
    (32, 4, 256, 32, [64, 777], 256),
    (16, 4, 64, 16, [1, 15, 17, 511, 513, 1300], 0),     # D = 64: two 64-byte rows per swizzled line
    (8, 1, 64, 32, [40, 700], 64),
    (32, 4, 64, 16, [3, 300], 0),                        # G = 8
    (32, 8, 128, 48, [47, 49, 1000], 480),               # three 16-token tiles per block
    (16, 4, 64, 80, [79, 81, 900], 400),                 # five tiles per block, token-pair lines
    (32, 8, 128, 16, [5000, 2049, 10], 0),               # the automatic E4M3 size: 2048-token partitions
]


@pytest.mark.parametrize("q_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", FP8_CASES)
def test_decode_fp8_matches_oracle(api, q_dtype, case):
    Hq, Hkv, D, b, lengths, part = case
    gen = torch.Generator().manual_seed(hash((Hq, Hkv, D, b, len(lengths), part)) & 0xFFFF)
    Kc, Vc, ks, vs, tables, lens = _fp8_setup(lengths, Hkv, D, b, gen)
    q = torch.randn((len(lengths), Hq, D), generator=gen).to(q_dtype)
    scale = 1 / math.sqrt(D)
    got = _decode(api, q, Kc, Vc, ks, vs, tables, lens, scale, part).double().numpy()
    want = _oracle(q, Kc, Vc, ks, vs, tables, lens, b, scale)
    assert np.abs(got - want).max() <= TOL[q_dtype]
    assert api.pa_get_device_error() == 0


def test_decode_fp8_nan_codes_in_unwritten_slots_are_masked(api):
    gen = torch.Generator().manual_seed(21)
    Kc, Vc, ks, vs, tables, lens = _fp8_setup([21], 2, 128, 16, gen)
    blk = int(tables[0, 1])
    Kc[blk, :, 5:] = 0x7F                                 # E4M3 NaN
    Vc[blk, :, 5:] = 0xFF
    q = torch.randn((1, 8, 128), generator=gen).half()
    got = _decode(api, q, Kc, Vc, ks, vs, tables, lens, 0.088)
    want = _oracle(q, Kc, Vc, ks, vs, tables, lens, 16, 0.088)
    assert torch.isfinite(got).all()
    assert np.abs(got.double().numpy() - want).max() <= 2e-3


def test_decode_fp8_d64_nan_codes_in_unwritten_slots_are_masked(api):
    """D = 64 (token pairs in one swizzled line): garbage past the length in the tail block,
    including the other token of a line, does not leak."""
    gen = torch.Generator().manual_seed(22)
    Kc, Vc, ks, vs, tables, lens = _fp8_setup([21], 2, 64, 16, gen)
    blk = int(tables[0, 1])
    Kc[blk, :, 5:] = 0x7F                                 # E4M3 NaN
    Vc[blk, :, 5:] = 0xFF
    q = torch.randn((1, 4, 64), generator=gen).half()
    got = _decode(api, q, Kc, Vc, ks, vs, tables, lens, 0.125)
    want = _oracle(q, Kc, Vc, ks, vs, tables, lens, 16, 0.125)
    assert torch.isfinite(got).all()
    assert np.abs(got.double().numpy() - want).max() <= 2e-3


def test_config3_fp8_full_size_sampled():
    """The long-context workload with E4M3 pools (the benchmark's --kv fp8 launch)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from oracle import driver as odriver
    from paged_kv_cache_66_gb300 import api
    from paged_kv_cache_66_gb300.replay import Replay
    from workload import configs
    wl = configs.config3()
    gpu = Replay(wl, device="cuda", kv="fp8")
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False, layers=[0], kv="fp8")
    ora.run_setup()
    rec = ora.run_step_ops(0)[-1]
    plan = gpu.plan_step(0)
    assert plan.slots.tolist() == rec["slots"] and plan.lens.tolist() == rec["lens"]
    outs = gpu.run_step(gpu.device_step(plan))
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    for layer, row in [(0, 0), (13, 6), (31, 3)]:
        want = ora.attend(rec, layer, rows=[row])[0]
        assert np.abs(outs[layer][row].double().cpu().numpy() - want).max() <= wl.tolerance


def test_config2_fp8_every_row_over_steps():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from oracle import driver as odriver
    from paged_kv_cache_66_gb300.replay import Replay
    from workload import configs
    wl = configs.config2(steps=6)
    gpu = Replay(wl, device="cuda", kv="fp8")
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False, kv="fp8")
    ora.run_setup()
    for s in range(6):
        rec = ora.run_step_ops(s)[-1]
        plan = gpu.plan_step(s)
        outs = gpu.run_step(gpu.device_step(plan))
    want = ora.attend(rec, 0)
    assert np.abs(outs[0].double().cpu().numpy() - want).max() <= wl.tolerance
