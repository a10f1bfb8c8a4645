"""Byte accounting of bench.py (CPU only): effective vs unique K/V bytes, algorithmic bytes.

Effective bytes count every sequence's history (a shared prefix once per sequence); unique
bytes count each pool block a decode touches once.
"""
from types import SimpleNamespace

import numpy as np

import bench
from workload import configs


def test_unique_counts_shared_blocks_once():
    wl = configs.config2()
    per_block = 2 * wl.Hkv * wl.b * wl.D * wl.elt
    # two sequences sharing their first two blocks; the second has one private block beyond
    tables = np.array([[5, 9, 0], [5, 9, 4]], dtype=np.int32)
    plan = SimpleNamespace(tables=tables, lens=np.array([20, 40], dtype=np.int32), uids=[0, 1])
    assert bench._unique_kv_bytes(wl, plan) == 3 * per_block          # blocks {5, 9, 4}
    assert bench._kv_bytes(wl, plan.lens) == 60 * 2 * wl.Hkv * wl.D * wl.elt
    # padding past ceil(L / b) is never counted
    plan.lens = np.array([16, 16], dtype=np.int32)
    assert bench._unique_kv_bytes(wl, plan) == 1 * per_block


def test_algorithmic_bytes_of_the_fused_launch_add_the_new_rows():
    wl = configs.config2()
    plan = SimpleNamespace(tables=np.zeros((2, 4), np.int32), lens=np.array([33, 64], np.int32), uids=[0, 1])
    plain = bench._alg_bytes_decode(wl, plan)
    fused = bench._alg_bytes_decode(wl, plan, fused=True)
    assert fused - plain == 4 * 2 * wl.Hkv * wl.D * wl.elt + 8 * 2
    assert plain == bench._kv_bytes(wl, plan.lens) + 2 * 2 * wl.Hq * wl.D * wl.elt + (3 + 4) * 4 + 4 * 2


def test_cpu_model_is_reported():
    assert isinstance(bench._cpu_model(), str) and bench._cpu_model()


def test_prefill_flop_count_is_the_brute_force_pair_count():
    """The prefill metric counts 4 D Hq FLOPs per (query row, visible key) pair; the closed form of
    the pair count equals a direct count of key positions k <= history + r over the chunk."""
    for batch, history, chunk in [(1, 0, 1), (2, 0, 7), (3, 5, 4), (2, 33, 17)]:
        wl = configs.prefill_config(batch=batch, history=history, chunk=chunk)
        brute = batch * sum(1 for r in range(chunk) for k in range(history + chunk) if k <= history + r)
        assert wl.causal_pairs() == brute
    # the benchmark's 8 x 1024 over 3072: 8 (1024 * 3072 + 1024 * 1025 / 2) = 29 364 224 pairs per head
    wl = configs.prefill_config()
    assert wl.causal_pairs() == 29_364_224
    assert 4 * wl.D * wl.Hq * wl.causal_pairs() == 481_103_446_016
