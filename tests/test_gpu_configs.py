"""The five seeded workloads end to end on the GPU against the oracle (needs a GPU).

Small workloads are mirrored completely by the oracle (its own pools, tables
and attention): the whole K/V pool must match bit for bit and every output
within the dtype tolerance.  At full size (configs 3, 4 and 5) the GPU runs
exactly what the benchmark times and the oracle replays the same ops with its
own block manager; then

  * the host plan (slots, copy pairs, lengths, tables) equals the oracle's at
    every step;
  * every slot a step wrote -- arrivals' prompts and each sequence's newest
    token, in every checked layer -- holds exactly the K and V rows the
    workload defines for that (owner, position) (torch.equal);
  * at checkpoints, every live position of every sequence, read through the
    oracle's tables, holds exactly its defined rows (so no write landed in a
    block that another sequence reads);
  * a copy-on-write destination equals its source block, all slots, K and V;
  * sampled outputs match the fp64 oracle within the dtype tolerance.

The oracle's content route draws its q and K/V values with the seeded
generator on the GPU (bit-identical to the host draw; tested below) and does
its arithmetic on the host in fp64.
"""
import numpy as np
import pytest
import torch

from oracle import driver as odriver
from workload import configs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _replay(wl, **kw):
    from paged_kv_cache_66_gb300.replay import Replay
    return Replay(wl, device="cuda", **kw)


def _check_plan(plan, rec):
    assert plan.slots.tolist() == rec["slots"]
    assert [tuple(p) for p in plan.pairs.tolist()] == [tuple(p) for p in rec["pairs"]]
    assert plan.lens.tolist() == rec["lens"]
    assert plan.tables.tolist() == [row[: plan.tables.shape[1]] for row in rec["tables"]]


def _max_err(out, want):
    return float(np.abs(out.double().cpu().numpy() - want).max())


def _written(wl, recs):
    """(slots, owners, positions) of every row the oracle's records of one step wrote."""
    slots, owners, pos = [], [], []
    for r in recs:
        if r["op"] == "write":
            uids = [r["uid"]] * len(r["slots"])
        elif r["op"] == "step":
            uids = r["uids"]
        else:
            continue
        slots += list(r["slots"])
        pos += list(r["positions"])
        owners += [wl.content_owner(u, p) for u, p in zip(uids, r["positions"])]
    return (np.asarray(slots, dtype=np.int64), np.asarray(owners, dtype=np.int64),
            np.asarray(pos, dtype=np.int64))


def _rows_at(pool, slots, b):
    s = torch.as_tensor(slots, device=pool.device)
    return pool[s // b, :, s % b, :]


def _check_written(gpu, wl, recs, layer_indices):
    """Every slot of the step holds the defined rows, bit for bit, in each listed layer slot."""
    slots, owners, pos = _written(wl, recs)
    for li in layer_indices:
        layer = gpu.layers[li]
        for kind, pools in (("k", gpu.k_pools), ("v", gpu.v_pools)):
            want = configs.kv_rows(wl, layer, kind, owners, pos, device="cuda")
            got = _rows_at(pools[li], slots, wl.b)
            assert torch.equal(got, want), (kind, layer)


def _check_live(gpu, ora, layer_indices, uids):
    """Every live position of each sequence, read through the oracle's table, holds its
    defined K and V rows, bit for bit."""
    wl, t = ora.wl, ora.t
    for u in uids:
        L = t.lengths[u]
        pos = np.arange(L, dtype=np.int64)
        blocks = np.asarray(t.tables[u], dtype=np.int64)[pos // wl.b]
        slots = blocks * wl.b + pos % wl.b
        owners = wl.content_owners(u, pos)
        for li in layer_indices:
            layer = gpu.layers[li]
            for kind, pools in (("k", gpu.k_pools), ("v", gpu.v_pools)):
                want = configs.kv_rows(wl, layer, kind, owners, pos, device="cuda")
                assert torch.equal(_rows_at(pools[li], slots, wl.b), want), (u, kind, layer)


def test_generator_is_bit_identical_on_host_and_device():
    """The oracle's content route may draw on the GPU: the draws must equal the host's."""
    owners = np.array([0, 3, 3, 900000, 17], dtype=np.int64)
    pos = np.array([0, 1, 77, 131071, 4096], dtype=np.int64)
    for dt in ("f16", "bf16", "f32"):
        wl = configs.config5(D=64, G=4, b=16, dtype="bf16", steps=1)
        wl.dtype = dt
        for kind in ("k", "v"):
            host = configs.kv_rows(wl, 0, kind, owners, pos)
            dev = configs.kv_rows(wl, 0, kind, owners, pos, device="cuda").cpu()
            assert host.dtype == dev.dtype and torch.equal(host, dev), (dt, kind)
        assert torch.equal(configs.q_rows(wl, 3, 199, [0, 5, 127]),
                           configs.q_rows(wl, 3, 199, [0, 5, 127], device="cuda").cpu()), dt


@pytest.mark.parametrize("steps", [1])
def test_config1_full_mirror(steps):
    from paged_kv_cache_66_gb300 import api
    wl = configs.config1()
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=True)
    ora.run_setup()
    rec = ora.run_step_ops(0)[-1]
    plan = gpu.plan_step(0)
    _check_plan(plan, rec)
    outs = gpu.run_step(gpu.device_step(plan))
    torch.cuda.synchronize()
    assert torch.equal(gpu.k_pools[0].cpu(), ora.k_pool[0])
    assert torch.equal(gpu.v_pools[0].cpu(), ora.v_pool[0])
    assert _max_err(outs[0], ora.attend(rec, 0)) <= wl.tolerance
    assert api.pa_get_device_error() == 0


def test_config2_full_mirror_64_steps():
    from paged_kv_cache_66_gb300 import api
    wl = configs.config2()
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=True)
    ora.run_setup()
    worst = 0.0
    for s in range(len(wl.step_ops)):
        rec = ora.run_step_ops(s)[-1]
        plan = gpu.plan_step(s)
        _check_plan(plan, rec)
        outs = gpu.run_step(gpu.device_step(plan))
        if s % 8 == 0 or s == len(wl.step_ops) - 1:
            worst = max(worst, _max_err(outs[0], ora.attend(rec, 0)))
    torch.cuda.synchronize()
    assert torch.equal(gpu.k_pools[0].cpu(), ora.k_pool[0])
    assert torch.equal(gpu.v_pools[0].cpu(), ora.v_pool[0])
    assert worst <= wl.tolerance, worst
    assert api.pa_get_device_error() == 0


def test_config3_full_size():
    """8 x 32768 tokens, 32 layers, fp16, 512-token partitions (the benchmark's launch):
    the newest rows of all 32 layers, every live position of 4 layers, and all 8
    sequences' outputs on those 4 layers."""
    from paged_kv_cache_66_gb300 import api
    wl = configs.config3()
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False, input_device="cuda")
    ora.run_setup()
    recs = ora.run_step_ops(0)
    rec = recs[-1]
    plan = gpu.plan_step(0)
    _check_plan(plan, rec)
    assert plan.lens.tolist() == [32768] * 8
    outs = gpu.run_step(gpu.device_step(plan))
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    _check_written(gpu, wl, recs, range(wl.layers))
    layers = [0, 11, 22, 31]
    _check_live(gpu, ora, layers, rec["uids"])
    for layer in layers:
        want = ora.attend(rec, layer)
        for r in range(8):
            assert _max_err(outs[layer][r], want[r]) <= wl.tolerance, (layer, r)


def test_config4_full_size_with_cow():
    """256 sequences over a shared 512-token prefix; sequence 0's append copies the
    partially filled shared block first."""
    from paged_kv_cache_66_gb300 import api
    wl = configs.config4()
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False, input_device="cuda")
    ora.run_setup()
    recs = ora.run_step_ops(0)
    rec = recs[-1]
    plan = gpu.plan_step(0)
    _check_plan(plan, rec)
    assert len(plan.pairs) == 1                       # sequence 0's copy-on-write
    src, dst = (int(x) for x in plan.pairs[0])
    assert ora.t.tables[0][31] == dst and ora.t.tables[1][31] == src
    before = [gpu.k_pools[0][src].clone(), gpu.v_pools[0][src].clone()]
    outs = gpu.run_step(gpu.device_step(plan))
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    # the shared block is untouched, and the copy is the whole block in K and in V (the
    # token sequence 0 appended at position 500 is the prefix owner's own row there)
    for pools, src_before in zip((gpu.k_pools, gpu.v_pools), before):
        assert torch.equal(pools[0][src], src_before)
        assert torch.equal(pools[0][dst], src_before)
    _check_written(gpu, wl, recs, [0])
    _check_live(gpu, ora, [0], rec["uids"])
    lens = np.array(plan.lens)
    rows = sorted({0, 1, 2, 64, 128, 200, 255, int(lens.argmax()), int(lens.argmin())})
    want = ora.attend(rec, 0, rows=rows)
    for i, r in enumerate(rows):
        assert _max_err(outs[0][r], want[i]) <= wl.tolerance, r


# The stated continuous-batching run: 200 steps, finish probability 0.01, 64-token arrivals.
# These combos cover head dims 64 / 128 / 256, groups 1 / 4 / 8, blocks 16 / 32 and both dtypes.
CONFIG5_FULL = [(64, 1, 16, "f16"), (64, 8, 32, "bf16"), (128, 4, 16, "bf16"), (128, 8, 32, "f16"),
                (256, 1, 32, "bf16"), (256, 8, 16, "f16"), (64, 4, 32, "f16"), (256, 4, 16, "bf16")]


@pytest.mark.parametrize("combo", CONFIG5_FULL)
def test_config5_200_steps(combo):
    from paged_kv_cache_66_gb300 import api
    D, G, b, dt = combo
    wl = configs.config5(D=D, G=G, b=b, dtype=dt)          # 200 steps, p_finish 0.01
    assert len(wl.step_ops) == 200
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False, input_device="cuda")
    ora.run_setup()
    arrivals = 0
    for s in range(len(wl.step_ops)):
        recs = ora.run_step_ops(s)
        rec = recs[-1]
        arrivals += sum(1 for r in recs if r["op"] == "write")
        plan = gpu.plan_step(s)
        _check_plan(plan, rec)
        outs = gpu.run_step(gpu.device_step(plan))
        _check_written(gpu, wl, recs, [0])
        if s % 25 == 0 or s == len(wl.step_ops) - 1:
            torch.cuda.synchronize()
            assert api.pa_get_device_error() == 0, s
            lens = np.array(plan.lens)
            rows = sorted({0, 64, 127, int(lens.argmax()), int(lens.argmin())})
            want = ora.attend(rec, 0, rows=rows)
            for i, r in enumerate(rows):
                assert _max_err(outs[0][r], want[i]) <= wl.tolerance, (combo, s, r)
        if s % 50 == 49:
            _check_live(gpu, ora, [0], rec["uids"])
    assert arrivals > 100, arrivals          # the pool really churned (~1.3 arrivals per step)


@pytest.mark.parametrize("combo", configs.CONFIG5_COMBOS)
def test_config5_sweep_short(combo):
    """All 36 combos, 6 steps at a high finish rate (arrivals in every few steps)."""
    from paged_kv_cache_66_gb300 import api
    D, G, b, dt = combo
    steps = 6
    wl = configs.config5(D=D, G=G, b=b, dtype=dt, steps=steps, p_finish=0.05)
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False, input_device="cuda")
    ora.run_setup()
    for s in range(steps):
        recs = ora.run_step_ops(s)
        rec = recs[-1]
        plan = gpu.plan_step(s)
        _check_plan(plan, rec)
        outs = gpu.run_step(gpu.device_step(plan))
        _check_written(gpu, wl, recs, [0])
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    lens = np.array(plan.lens)
    rows = sorted({0, 64, 127, int(lens.argmax()), int(lens.argmin())})
    want = ora.attend(rec, 0, rows=rows)
    for i, r in enumerate(rows):
        assert _max_err(outs[0][r], want[i]) <= wl.tolerance, (combo, r)
