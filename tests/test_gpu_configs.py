"""The five seeded workloads end to end on the GPU against the oracle (needs a GPU).

Small workloads are mirrored completely by the oracle (its own pools, tables
and attention): the whole K/V pool must match bit for bit and every output
within the dtype tolerance.  At full size (configs 3, 4 and the config-5
sweep) the GPU runs exactly what the benchmark times and the oracle checks
sampled (sequence, layer) outputs from the token contents the workload
defines, plus the host tables step by step.
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


def test_config3_full_size_sampled():
    """8 x 32768 tokens, 32 layers, fp16, 512-token partitions (the benchmark's launch)."""
    from paged_kv_cache_66_gb300 import api
    wl = configs.config3()
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False, layers=[0])
    ora.run_setup()
    rec = ora.run_step_ops(0)[-1]
    plan = gpu.plan_step(0)
    _check_plan(plan, rec)
    assert plan.lens.tolist() == [32768] * 8
    outs = gpu.run_step(gpu.device_step(plan))
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    for layer, row in [(0, 0), (17, 5), (31, 7)]:
        ora.layers = [layer]
        want = ora.attend(rec, layer, rows=[row])[0]
        assert _max_err(outs[layer][row], want) <= wl.tolerance


def test_config4_full_size_sampled_with_cow():
    from paged_kv_cache_66_gb300 import api
    wl = configs.config4()
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False)
    ora.run_setup()
    rec = ora.run_step_ops(0)[-1]
    plan = gpu.plan_step(0)
    _check_plan(plan, rec)
    assert len(plan.pairs) == 1                       # sequence 0's copy-on-write
    src, dst = (int(x) for x in plan.pairs[0])
    before_src = gpu.k_pools[0][src].clone()
    outs = gpu.run_step(gpu.device_step(plan))
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    # the shared block is untouched; the copy holds its first 4 slots plus the new token
    assert torch.equal(gpu.k_pools[0][src], before_src)
    assert torch.equal(gpu.k_pools[0][dst][:, :4], before_src[:, :4])
    lens = np.array(plan.lens)
    rows = [0, 1, int(lens.argmax()), int(lens.argmin()), 128, 255]
    want = ora.attend(rec, 0, rows=rows)
    for i, r in enumerate(rows):
        assert _max_err(outs[0][r], want[i]) <= wl.tolerance, r


@pytest.mark.parametrize("combo", configs.CONFIG5_COMBOS)
def test_config5_sweep_sampled(combo):
    from paged_kv_cache_66_gb300 import api
    D, G, b, dt = combo
    steps = 6
    wl = configs.config5(D=D, G=G, b=b, dtype=dt, steps=steps, p_finish=0.05)
    gpu = _replay(wl)
    gpu.run_setup()
    ora = odriver.OracleRun(wl, pools=False)
    ora.run_setup()
    for s in range(steps):
        rec = ora.run_step_ops(s)[-1]
        plan = gpu.plan_step(s)
        _check_plan(plan, rec)
        outs = gpu.run_step(gpu.device_step(plan))
    torch.cuda.synchronize()
    assert api.pa_get_device_error() == 0
    lens = np.array(plan.lens)
    rows = sorted({0, 64, 127, int(lens.argmax()), int(lens.argmin())})
    want = ora.attend(rec, 0, rows=rows)
    for i, r in enumerate(rows):
        assert _max_err(outs[0][r], want[i]) <= wl.tolerance, (combo, r)
