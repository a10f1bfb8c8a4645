"""C-ABI library checks and the C++ host block manager against the oracle (CPU only).

The library is built for sm_103a and loaded with ctypes; nothing here launches
a kernel: host-manager entry points run on the CPU, and device entry points
are only called with arguments that their host-side validation rejects.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

from oracle import blocks as oblocks
from oracle import driver as odriver
from paged_kv_cache_66_gb300 import _lib
from paged_kv_cache_66_gb300.host import HostBlockManager
from tests.conftest import ROOT, golden
from workload import configs


def _declared_functions():
    names = []
    for h in ("pagedkv.h", "pagedkv_host.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(pa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = _declared_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


@pytest.mark.parametrize("header", ["pagedkv.h", "pagedkv_host.h"])
@pytest.mark.parametrize("lang", ["c", "c++"])
def test_public_headers_compile_standalone(header, lang, tmp_path):
    """Each public header is self-contained, warning-free C11 and C++17 (no CUDA or torch types)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip(f"no {lang} compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text(f'#include "{header}"\n')
    std = "-std=c11" if lang == "c" else "-std=c++17"
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    code = re.sub(r"/\*.*?\*/|//[^\n]*", "", open(os.path.join(ROOT, "include", header)).read(), flags=re.S)
    assert not re.search(r"#include\s*[<\"](cuda|torch|ATen)|\bcuda\w*_t\b|\bCU\w+\b|\btorch\b|\bat::", code)


def test_status_strings():
    lib = _lib.load()
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.pa_status_string(code).decode() == name


def test_device_entry_points_validate_before_touching_cuda():
    lib = _lib.load()
    null = C.c_void_p(0)
    # null pools
    assert lib.pa_kv_append(null, null, null, null, null, 4, 16, 2, 64, 16, 1, null) == 1
    # unknown dtype
    assert lib.pa_kv_append(null, null, null, null, null, 4, 16, 2, 64, 16, 7, null) == 1
    # unsupported head_dim / group / block size for decode, nothing launched
    assert lib.pa_decode(null, null, null, null, 16, null, 4, null, 2, 4, 2, 96, 16, 0.1, 0, null, 0, 1,
                         null) == 2
    assert lib.pa_decode(null, null, null, null, 16, null, 4, null, 2, 6, 2, 64, 16, 0.1, 0, null, 0, 1,
                         null) == 2
    assert lib.pa_decode(null, null, null, null, 16, null, 4, null, 2, 4, 2, 64, 24, 0.1, 0, null, 0, 1,
                         null) == 2
    # Hq not a multiple of Hkv; partition not a multiple of the block size
    assert lib.pa_decode(null, null, null, null, 16, null, 4, null, 2, 5, 2, 64, 16, 0.1, 0, null, 0, 1,
                         null) == 1
    assert lib.pa_decode(null, null, null, null, 16, null, 4, null, 2, 4, 2, 64, 32, 0.1, 48, null, 0, 1,
                         null) == 1
    # null tensors
    assert lib.pa_decode(null, null, null, null, 16, null, 4, null, 2, 4, 2, 64, 16, 0.1, 0, null, 0, 1,
                         null) == 1
    # prefill: f32 and D = 96 unsupported; Hq not a multiple of Hkv; null tensors; empty batch is a no-op
    #            out   q     kp    vp    N   tbl  mb  lens  qst   B  T  mq Hq Hkv D   b   scale dtype
    assert lib.pa_prefill(null, null, null, null, 16, null, 4, null, null, 2, 8, 4, 4, 2, 64, 16, 0.1, 0,
                          null) == 2
    assert lib.pa_prefill(null, null, null, null, 16, null, 4, null, null, 2, 8, 4, 4, 2, 96, 16, 0.1, 1,
                          null) == 2
    assert lib.pa_prefill(null, null, null, null, 16, null, 4, null, null, 2, 8, 4, 5, 2, 64, 16, 0.1, 1,
                          null) == 1
    assert lib.pa_prefill(null, null, null, null, 16, null, 4, null, null, 2, 8, 4, 4, 2, 64, 16, 0.1, 1,
                          null) == 1
    assert lib.pa_prefill(null, null, null, null, 16, null, 4, null, null, 0, 0, 0, 4, 2, 64, 16, 0.1, 1,
                          null) == 0
    ptrs = (C.c_void_p * 1)(None)
    assert lib.pa_copy_blocks(ptrs, ptrs, 1, null, 1, 16, 4096, null) == 1
    assert lib.pa_copy_blocks(ptrs, ptrs, 1, null, 1, 16, 4095, null) == 1


def test_workspace_size():
    lib = _lib.load()
    # one partition: no workspace
    assert lib.pa_decode_workspace_size(8, 32, 128, 32, 16, 512) == 0
    # 8 x 32 heads x 64 partitions: (max, normaliser) + 128 partial floats each
    rows = 8 * 32 * 64
    ml = (rows * 8 + 255) // 256 * 256
    assert lib.pa_decode_workspace_size(8, 32, 128, 2048, 16, 512) == ml + rows * 128 * 4
    assert lib.pa_decode_workspace_size(8, 32, 128, 2048, 16, 0) == ml + rows * 128 * 4


def test_auto_partition_size():
    """partition_tokens = 0: 512 tokens, halved down to 128 while batch * ceil(Hq / 8) *
    partitions stays under 608.  Checked through the workspace size, which uses the same rule."""
    lib = _lib.load()

    def same(shape, part):
        return lib.pa_decode_workspace_size(*shape, 0) == lib.pa_decode_workspace_size(*shape, part)

    def units(B, Hq, mb, b, part):
        return B * -(-Hq // 8) * -(-mb * b // part)

    # the long-context batch keeps 512 (8 x 4 x 64 units)
    assert same((8, 32, 128, 2048, 16), 512) and units(8, 32, 2048, 16, 512) >= 608
    # the Llama-3-8B-shaped batch of 32 histories under ~530 tokens: 512 -> 256 -> 128
    assert units(32, 32, 34, 16, 512) < 608 and units(32, 32, 34, 16, 256) < 608
    assert same((32, 32, 128, 34, 16), 128) and not same((32, 32, 128, 34, 16), 512)
    # large batches keep 512; b = 256 stops at 256 (a partition is a multiple of b)
    assert same((128, 32, 64, 270, 16), 512)
    assert same((1, 8, 128, 4, 256), 256)
    # b = 48: 480 tokens (the largest multiple of 48 up to 512), then 240
    assert same((64, 32, 128, 40, 48), 480) and same((1, 8, 128, 40, 48), 240)


def test_kernel_choices_accept_the_declared_values_only():
    """pa_set_decode_kernel / pa_set_decode_heads_per_cta store a process-wide choice
    (host only): the enum values of include/pagedkv.h are taken, others refused."""
    lib = _lib.load()
    for k in (0, 1, 2):
        assert lib.pa_set_decode_kernel(k) == 0
    assert lib.pa_set_decode_kernel(3) == 1
    for h in (0, 1, 2):
        assert lib.pa_set_decode_heads_per_cta(h) == 0
    assert lib.pa_set_decode_heads_per_cta(3) == 1 and lib.pa_set_decode_heads_per_cta(-1) == 1
    assert lib.pa_set_decode_kernel(0) == 0
    assert lib.pa_set_decode_heads_per_cta(0) == 0


# ------------------------------------------------------------------ host manager

def test_host_slot_example_and_exceptions():
    g = golden("p1_slot_example.json")
    b = g["block_size"]
    order = [5, 1, 7] + [x for x in range(8) if x not in (5, 1, 7)]
    h = HostBlockManager(8, b, order)
    h.create(0)
    h.reserve(0, 12)
    assert h.table(0) == g["table"]
    slot = int(h.slots(0, g["position"], 1)[0])
    assert divmod(slot, b) == tuple(g["expected_block_offset"])
    with pytest.raises(ValueError):
        h.create(0)
    with pytest.raises(KeyError):
        h.reserve(99, 1)
    h.advance(0, 12)
    with pytest.raises(MemoryError):
        h.create(1) or h.reserve(1, 100)
    assert h.length(1) == 0 and h.table(1) == []      # all-or-nothing


def test_host_over_release_is_reported():
    h = HostBlockManager(4, 4)
    h.create(0)
    h.reserve(0, 4)
    h.advance(0, 4)
    h.fork(0, 1)
    h.free(0)
    h.free(1)
    assert h.num_free == 4
    with pytest.raises(KeyError):
        h.free(1)


def test_host_fork_cow_p1_numbers():
    g = golden("p1_fork_cow.json")
    h = HostBlockManager(64, g["block_size"])
    h.create(100)
    h.reserve(100, g["prompt_tokens"])
    h.advance(100, g["prompt_tokens"])
    used0 = 64 - h.num_free
    for i in range(g["forks"]):
        h.fork(100, i)
    used1 = 64 - h.num_free
    for i in range(g["forks"]):
        assert len(h.reserve(i, 1)) == 1
        h.advance(i, 1)
    used2 = 64 - h.num_free
    e = g["expected"]
    assert (used0, used1 - used0, used2 - used1) == (e["parent_blocks"], e["new_blocks_after_4_forks"],
                                                      e["new_blocks_after_each_sample_writes_a_token"])


def test_host_prefix_sharing_p2_numbers():
    g = golden("p2_prefix_sharing.json")
    e = g["expected"]
    h = HostBlockManager(1024, g["block_size"])
    h.create(-1)
    h.reserve(-1, g["system_prompt_tokens"])
    h.advance(-1, g["system_prompt_tokens"])
    for i in range(g["forks"]):
        h.fork(-1, i)
        for _ in range(g["tokens_per_fork"]):
            h.reserve(i, 1)
            h.advance(i, 1)
    assert len(set(h.table(0)) & set(h.table(1))) == e["shared_blocks"]
    assert 1024 - h.num_free == e["blocks_used"]
    h.free(-1)
    assert 1024 - h.num_free == e["used_after_base_free"]
    for i in range(g["forks"]):
        h.free(i)
    assert 1024 - h.num_free == e["used_after_all_free"]


def test_host_prefix_cache_p1_numbers():
    g = golden("p1_prefix_cache.json")
    e = g["expected"]
    h = HostBlockManager(256, g["block_size"])
    shared = list(range(1000, 1000 + g["shared_tokens"]))
    prefilled = 0
    for r in range(g["requests"]):
        prompt = shared + [r * 100 + i for i in range(g["own_tokens"])]
        reused = h.prefix_attach(r, prompt)
        h.reserve(r, len(prompt) - reused)
        h.advance(r, len(prompt) - reused)
        h.prefix_remember(r, prompt)
        prefilled += len(prompt) - reused
    assert prefilled == e["tokens_prefilled"]
    assert 256 - h.num_free == e["blocks_in_use"]


def _mirror(seed, ops=3000, N=48, b=4):
    """Random op streams applied to the C++ manager and the oracle side by side."""
    r = np.random.default_rng(seed)
    order = r.permutation(N)
    h = HostBlockManager(N, b, order)
    o = oblocks.SeqTables(N, b, order)
    opc = oblocks.PrefixTable(o)
    live, nxt = [], 0
    for _ in range(ops):
        kind = int(r.integers(0, 8))
        try:
            if kind == 0 or not live:
                res_o = o.create(nxt)
                h.create(nxt)
                live.append(nxt)
                nxt += 1
            elif kind in (1, 2):
                s = live[int(r.integers(len(live)))]
                n = int(r.integers(1, 7))
                try:
                    po = o.reserve(s, n)
                except MemoryError:
                    with pytest.raises(MemoryError):
                        h.reserve(s, n)
                    continue
                ph = h.reserve(s, n)
                assert ph == po
                o.advance(s, n)
                h.advance(s, n)
            elif kind == 3:
                s = live[int(r.integers(len(live)))]
                o.fork(s, nxt)
                h.fork(s, nxt)
                live.append(nxt)
                nxt += 1
            elif kind == 4:
                s = live.pop(int(r.integers(len(live))))
                o.free(s)
                h.free(s)
            elif kind == 5:
                s = live[int(r.integers(len(live)))]
                L = int(r.integers(0, o.lengths[s] + 1))
                o.truncate(s, L)
                h.truncate(s, L)
            elif kind == 6:
                prompt = [int(x) for x in r.integers(0, 3, size=int(r.integers(1, 14)))]
                a = opc.attach(nxt, prompt)
                assert h.prefix_attach(nxt, prompt) == a
                live.append(nxt)
                nxt += 1
                s = live[-1]
                n = len(prompt) - a
                try:
                    o.reserve(s, n)
                except MemoryError:
                    with pytest.raises(MemoryError):
                        h.reserve(s, n)
                    continue
                h.reserve(s, n)
                o.advance(s, n)
                h.advance(s, n)
                opc.remember(s, prompt)
                h.prefix_remember(s, prompt)
            else:
                want = int(r.integers(0, N))
                opc.evict(want)
                h.prefix_evict(want)
        except MemoryError:
            pass
        assert h.num_free == o.allocator.num_free
        assert h.prefix_entries == len(opc.entries)
    for s in live:
        assert h.table(s) == o.tables[s] and h.length(s) == o.lengths[s]
    for blk in range(N):
        assert h.refcount(blk) == o.allocator.refs[blk]


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_host_manager_matches_oracle_random_ops(seed):
    _mirror(seed)


def _host_replay(wl):
    """Replay a workload's host ops on the C++ manager; yield step records."""
    h = HostBlockManager(wl.num_blocks, wl.b, wl.free_order)

    def apply(op):
        k = op[0]
        if k == "create":
            h.create(op[1])
        elif k == "write":
            s = h.length(op[1])
            pairs = h.reserve(op[1], op[2])
            slots = h.slots(op[1], s, op[2]).tolist()
            h.advance(op[1], op[2])
            return {"pairs": pairs, "slots": slots}
        elif k == "fork":
            h.fork(op[1], op[2])
        elif k == "truncate":
            h.truncate(op[1], op[2])
        elif k == "free":
            h.free(op[1])
        elif k == "step":
            uids = list(op[1])
            stride = max(len(h.table(u)) for u in uids) + 1
            tables = np.zeros((len(uids), stride), np.int32)
            lens = np.zeros(len(uids), np.int32)
            slots = np.zeros(len(uids), np.int64)
            pairs, w = h.decode_step(uids, tables, lens, slots)
            return {"pairs": [tuple(map(int, p)) for p in pairs], "slots": slots.tolist(),
                    "tables": tables[:, :w].tolist(), "lens": lens.tolist()}
        return {}

    out = [apply(op) for op in wl.setup_ops]
    for ops in wl.step_ops:
        out += [apply(op) for op in ops]
    return out


@pytest.mark.parametrize("make", [lambda: configs.config1(), lambda: configs.config2(steps=8),
                                  lambda: configs.config3(layers=1, steps=20),
                                  lambda: configs.config4(),
                                  lambda: configs.config5(D=128, G=4, b=16, dtype="bf16", steps=60),
                                  lambda: configs.config5(D=64, G=8, b=32, dtype="f16", steps=60)])
def test_host_replay_matches_oracle_bit_exact(make):
    wl = make()
    got = _host_replay(wl)
    o = odriver.OracleRun(wl, pools=False)
    want = o.run_setup()
    for s in range(len(wl.step_ops)):
        want += o.run_step_ops(s)
    assert len(got) == len(want)
    for g, w in zip(got, want):
        for key in g:
            assert g[key] == [tuple(x) for x in w[key]] if key == "pairs" else g[key] == w[key], key


def test_decode_tile_to_table_entry_is_exact_over_the_accepted_shapes():
    """The tensor-core decode finds tile i's table entry as (i * ceil(65536 / t)) >> 16 with
    t = b / 16 tiles per block, instead of dividing.  The limits the C ABI accepts (partition
    tokens, block size) bound i and t; the quotient must be exact over all of them."""
    api_src = open(os.path.join(ROOT, "paged_kv_cache_66_gb300", "csrc", "pa_api.cu")).read()
    kern_src = open(os.path.join(ROOT, "paged_kv_cache_66_gb300", "csrc", "decode_mma.cuh")).read()
    launch_src = open(os.path.join(ROOT, "paged_kv_cache_66_gb300", "csrc", "pa_launch.h")).read()
    assert "constexpr int kMaxPartition = pa::kMaxPartitionTokens;" in api_src
    max_part = int(re.search(r"constexpr int kMaxPartitionTokens = (\d+);", launch_src).group(1))
    max_b = int(re.search(r"block_size % 16 != 0 \|\| block_size > (\d+)\) return PA_ERR_UNSUPPORTED", api_src).group(1))
    assert "(65536u + tpb - 1) / tpb" in kern_src and "* inv_tpb) >> 16" in kern_src
    i = np.arange(max_part // 16, dtype=np.uint64)
    for t in range(1, max_b // 16 + 1):
        inv = (65536 + t - 1) // t
        assert np.array_equal((i * np.uint64(inv)) >> np.uint64(16), i // np.uint64(t)), t
        assert int(i[-1]) * inv < 2**32  # the product stays within the kernel's 32-bit unsigned
