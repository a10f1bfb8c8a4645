"""The N > 1 path of the benchmark on CPU: two gloo ranks, one replica each.

The path shards by sequence with no exchange, so multi-GPU runs are
independent replicas: each rank plans its own steps with its own host block
manager; the only communication is the barrier and the max / sum of the timed
region and the bytes (bench.py's helpers), checked here with world size 2.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from paged_kv_cache_66_gb300.host import HostBlockManager
    from workload import configs

    wl = configs.config3(steps=4, layers=1)
    h = HostBlockManager(wl.num_blocks, wl.b, wl.free_order)
    for op in wl.setup_ops:
        if op[0] == "create":
            h.create(op[1])
        else:
            h.reserve(op[1], op[2])
            h.advance(op[1], op[2])
    uids = list(wl.step_ops[0][-1][1])
    stride = max(len(h.table(u)) for u in uids) + 4
    tables = np.zeros((len(uids), stride), np.int32)
    lens = np.zeros(len(uids), np.int32)
    slots = np.zeros(len(uids), np.int64)
    kv = 0
    for _ in range(4):
        h.decode_step(uids, tables, lens, slots)
        kv += bench._kv_bytes(wl, lens)
    bench._barrier(world)
    t_max = bench._max_over_ranks(1.0 + rank, world, "cpu")          # rank r "took" 1 + r ms
    kv_all = bench._sum_over_ranks(float(kv), world, "cpu")
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), tables=tables, lens=lens, slots=slots, t_max=t_max,
             kv_all=kv_all, kv=kv)
    dist.destroy_process_group()


def test_two_gloo_ranks_run_identical_replicas(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npz")
    r1 = np.load(tmp_path / "rank1.npz")
    for k in ("tables", "lens", "slots"):
        assert np.array_equal(r0[k], r1[k])           # independent replicas of the same workload
    assert float(r0["t_max"]) == float(r1["t_max"]) == 2.0   # max over ranks
    assert float(r0["kv_all"]) == float(r1["kv_all"]) == 2 * float(r0["kv"])
    assert list(r0["lens"]) == [32767 + 4] * 8
