"""The seeded input generator and the oracle's op replay (CPU only)."""
import numpy as np
import torch

from oracle import attention, driver
from workload import configs, rng


def test_mix32_tensor_matches_python_int():
    xs = [0, 1, 2, 0xDEADBEEF, 0xFFFFFFFF, 123456789, 2**31]
    got = rng.mix32(torch.tensor(xs, dtype=torch.int64)).tolist()
    assert got == [rng.mix32_int(x) for x in xs]


def test_values_deterministic_and_unit_normalish():
    key = rng.stream_key(3, 1, 2)
    idx = torch.arange(1 << 18, dtype=torch.int64) * 7919 + (1 << 40)
    a = rng.normal_from_index(key, idx)
    b = rng.normal_from_index(key, idx.clone())
    assert torch.equal(a, b)
    assert abs(a.mean().item()) < 0.01 and abs(a.std().item() - 1.0) < 0.01
    assert a.abs().max().item() < 3.47
    # a different stream gives different values
    c = rng.normal_from_index(rng.stream_key(3, 1, 3), idx)
    assert not torch.equal(a, c)


def test_kv_rows_are_addressed_by_content():
    wl = configs.config2()
    a = configs.kv_rows(wl, 0, "k", [5, 5, 6], [10, 11, 10])
    b = configs.kv_rows(wl, 0, "k", [5], [11])
    assert torch.equal(a[1], b[0]) and not torch.equal(a[0], a[2])
    sub = configs.kv_rows(wl, 0, "k", [5], [11], heads=[3, 1])
    assert torch.equal(sub[0, 0], b[0, 3]) and torch.equal(sub[0, 1], b[0, 1])
    assert a.dtype == torch.bfloat16


def test_configs_shapes():
    c = configs.all_configs()
    w1 = c[1]()
    assert (w1.Hq, w1.Hkv, w1.D, w1.b, w1.dtype, w1.num_blocks) == (4, 2, 64, 16, "f32", 16)
    w3 = c[3](layers=2)
    assert w3.num_blocks == 20000 and w3.partition_tokens == 512
    w4 = c[4]()
    assert sum(1 for op in w4.setup_ops if op[0] == "fork") == 255
    w5 = c[5](D=64, G=8, b=32, dtype="f16", steps=20)
    assert w5.Hkv == 4 and w5.num_blocks == 16384 and len(w5.step_ops) == 20
    assert len(configs.CONFIG5_COMBOS) == 36


def test_config1_replay_pool_route_equals_content_route():
    """Attention gathered through the oracle's own pool and tables equals
    attention over the per-position token contents (two independent routes)."""
    wl = configs.config1()
    a = driver.OracleRun(wl, pools=True)
    b = driver.OracleRun(wl, pools=False)
    a.run_setup(); b.run_setup()
    ra = a.run_step_ops(0)[-1]
    rb = b.run_step_ops(0)[-1]
    assert ra["tables"] == rb["tables"] and ra["slots"] == rb["slots"]
    assert ra["lens"] == [2, 8, 17, 34]
    oa, ob = a.attend(ra, 0), b.attend(rb, 0)
    assert np.array_equal(oa, ob)
    # and the split/merge cross-check agrees with the definition on this data
    q = configs.q_rows(wl, 0, 0, [3]).double().numpy()[0]
    K, V = b.history(3, 34, 0)
    np.testing.assert_allclose(attention.decode_attention_split(q, K, V, wl.scale, 16, 16),
                               ob[3], atol=1e-13)


def test_config4_prefix_cow_replay():
    wl = configs.config4(batch=8, num_blocks=512)
    run = driver.OracleRun(wl, pools=True)
    run.run_setup()
    prefix = run.t.tables[1][:32]
    assert all(run.t.tables[u][:32] == prefix for u in range(8))
    assert all(run.t.allocator.refs[blk] == 8 for blk in prefix)
    rec = run.run_step_ops(0)[-1]
    assert len(rec["pairs"]) == 1 and rec["pairs"][0][0] == prefix[31]
    assert rec["lens"][0] == 501
    # pool route and content route agree (the copy-on-write kept both views right)
    b = driver.OracleRun(wl, pools=False)
    b.run_setup()
    rb = b.run_step_ops(0)[-1]
    assert np.array_equal(run.attend(rec, 0), b.attend(rb, 0))


def test_config5_small_replay_with_churn():
    wl = configs.config5(D=64, G=4, b=16, dtype="f16", steps=30, batch=16, p_finish=0.1,
                         prompt=8)
    run = driver.OracleRun(wl, pools=True)
    run.run_setup()
    recs = []
    for s in range(30):
        recs.append(run.run_step_ops(s)[-1])
    frees = sum(1 for ops in wl.step_ops for op in ops if op[0] == "free")
    assert frees > 0
    b = driver.OracleRun(wl, pools=False)
    b.run_setup()
    for s in range(30):
        rb = b.run_step_ops(s)[-1]
    assert np.array_equal(run.attend(recs[-1], 0), b.attend(rb, 0))
