"""Benchmark of paged decode on GB300: one JSON line on stdout.

A step is one pass of the whole hot path over one batch: host table/slot
resolution and copy-on-write decisions (C++ block manager), then on the
device pa_copy_blocks, and per layer pa_kv_append of arrivals' prompts and one
pa_decode_append (each sequence's new row + decode + merge).  The default
workload is the long-context decode: 8 sequences x 32768 tokens, 32 layers of
independent K/V, fp16, Hq 32 / Hkv 8 / D 128, b 16, 512-token partitions.

  value   effective KV GB/s of the device path: sum over layers and sequences of
          L * 2 * Hkv * D * sizeof(dtype) bytes per step / device step time.
          The host plans of all timed steps are made and uploaded before the
          timed region (inputs resident in HBM).
  e2e     the same metric through the public API with host buffers: the C++
          plan of each step, host->device copies of its q / new K / new V rows
          and tables, the kernels, and the device->host copy of every layer's
          output, all inside the timed region.
  --impl reference   times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workload import configs as wcfg  # noqa: E402

METRIC = "paged decode-attn KV GB/s (% of GB300 HBM peak); seq-steps/s at batch×context"
KERNEL_SOURCES = ["paged_kv_cache_66_gb300/csrc/decode_mma.cuh", "paged_kv_cache_66_gb300/csrc/decode_merge.cuh",
                  "paged_kv_cache_66_gb300/csrc/pa_common.cuh"]


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t)
    return float(t.item())


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """Dense 16-bit tensor peak for a kernel timed alone: the measured cuBLAS bf16
    burst figure (fp16 runs at the same nominal rate)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except Exception:
        return 1900.0, "fallback bf16 burst"


def _kernel_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _launch_key(args, wl, rp) -> str:
    """Name of the profiled launch: the workload plus whatever changes the kernel or its bytes."""
    key = wl.name
    if args.kv == "fp8":
        key += "+e4m3"
    if rp.partition_tokens != wl.partition_tokens:
        key += f"+p{rp.partition_tokens}"
    if args.kernel != "auto":
        key += f"+{args.kernel}"
    if args.unfused and args.kv == "native":
        key += "+unfused"
    return key


def _profiled_traffic(workload: str):
    """dram bytes per launch from a committed ncu summary, if taken on this kernel source."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    sha = _kernel_sha()
    for name in sorted(os.listdir(d)):
        if not name.endswith(".md"):
            continue
        txt = open(os.path.join(d, name)).read()
        m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
        m_wl = re.search(r"bench_workload:\s*(\S+)", txt)
        if m_sha and m_tr and m_wl and m_sha.group(1) == sha and m_wl.group(1) == workload:
            return float(m_tr.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": n}


def _workload(cfg: int, steps: int, combo=None):
    if cfg == 3:
        return wcfg.config3(steps=steps)
    if cfg == 2:
        return wcfg.config2(steps=steps)
    if cfg == 4:
        return wcfg.config4(steps=steps)
    if cfg == 5:
        D, G, b, dt = combo
        return wcfg.config5(D=D, G=G, b=b, dtype=dt, steps=steps)
    return wcfg.config1()


def _kv_bytes(wl, lens, elt=None) -> int:
    """Effective K/V bytes one decode reads: sum of L * 2 * Hkv * D * (stored element size)."""
    return int(np.sum(np.asarray(lens, dtype=np.int64))) * 2 * wl.Hkv * wl.D * (wl.elt if elt is None else elt)


def _unique_kv_bytes(wl, plan, elt=None) -> int:
    """Unique K/V bytes one decode touches: distinct pool blocks in the batch's tables (a block
    shared by many sequences counted once) x 2 * Hkv * b * D * (stored element size)."""
    blocks = set()
    for row, L in zip(np.asarray(plan.tables), np.asarray(plan.lens, dtype=np.int64)):
        blocks.update(int(x) for x in row[: (int(L) + wl.b - 1) // wl.b])
    return len(blocks) * 2 * wl.Hkv * wl.b * wl.D * (wl.elt if elt is None else elt)


def _cpu_model() -> str:
    """CPU model name from /proc/cpuinfo (x86 'model name'; Arm implementer / part), else the machine."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    m = re.search(r"^model name\s*:\s*(.+)$", info, flags=re.M)
    if m:
        return m.group(1).strip()
    impl = re.search(r"^CPU implementer\s*:\s*(\S+)", info, flags=re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", info, flags=re.M)
    if impl and part:
        return f"{platform.machine()} implementer {impl.group(1)} part {part.group(1)}"
    return platform.machine()


def _alg_bytes_decode(wl, plan, kv_elt=None, fused=False) -> int:
    """Algorithmic bytes of one pa_decode launch: K/V history + q + out + block
    tables + lengths (scratch traffic of the split is not algorithmic).  A fused
    pa_decode_append also reads each sequence's new K/V row and its slot and
    writes the row into the pool."""
    B = len(plan.uids)
    tbl = int(np.sum((np.asarray(plan.lens, dtype=np.int64) + wl.b - 1) // wl.b)) * 4
    extra = (4 * B * wl.Hkv * wl.D * wl.elt + 8 * B) if fused else 0
    return _kv_bytes(wl, plan.lens, kv_elt) + 2 * B * wl.Hq * wl.D * wl.elt + tbl + 4 * B + extra


# ------------------------------------------------------------------ reference arm (CPU oracle)

def run_reference(args, ws, rank):
    if rank != 0:
        return
    from oracle import attention as oatt
    from oracle import driver as odriver
    # Bounded sample: one sequence of layer 0 per step, the oracle gathering the
    # history through its own pool and table, then the fp64 definition.  For the
    # long-context workload only the sampled sequence is built.
    wl = wcfg.config3(steps=1, layers=1, batch=1) if args.config == 3 else _workload(args.config, 1, args.combo)
    ora = odriver.OracleRun(wl, pools=True, layers=[0])
    ora.run_setup()
    rec = ora.run_step_ops(0)[-1]
    q = wcfg.q_rows(wl, 0, rec["step"], list(range(len(rec["uids"])))).double().numpy()
    B = len(rec["uids"])

    def one(i):
        r = i % B
        t0 = time.perf_counter()
        oatt.paged_decode(q[r], ora.k_pool[0], ora.v_pool[0], rec["tables"][r], rec["lens"][r], wl.b, wl.scale)
        return time.perf_counter() - t0, _kv_bytes(wl, [rec["lens"][r]])

    for i in range(args.warmup):
        one(i)
    tt, bb = 0.0, 0
    for i in range(args.steps):
        t, b = one(args.warmup + i)
        tt += t
        bb += b
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    val = bb / tt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "sample": "one sequence of layer 0 per step"},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu_model": _cpu_model(),
                             "sample": f"one {wl.name} sequence x layer 0 per step, {args.steps} steps"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(wl, budget_s: float = 15.0):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    from oracle import attention as oatt
    from workload import configs as wc
    L = int(wl.setup_ops[1][2]) + 1 if wl.setup_ops[1][0] == "write" else 4096
    L = min(L, 32768)
    # a single-sequence pool built from the workload's token contents
    nb = -(-L // wl.b)
    t0 = time.perf_counter()
    pos = np.arange(L, dtype=np.int64)
    owners = wl.content_owners(0, pos)
    k = wc.kv_rows(wl, 0, "k", owners, pos)
    v = wc.kv_rows(wl, 0, "v", owners, pos)
    perm = np.random.default_rng(0).permutation(nb)
    kp = torch.zeros((nb, wl.Hkv, wl.b, wl.D), dtype=wl.torch_dtype)
    vp = torch.zeros_like(kp)
    from oracle import cache_ops
    slots = perm[pos // wl.b] * wl.b + pos % wl.b
    cache_ops.append(kp, vp, k, v, slots, wl.b)
    q = wc.q_rows(wl, 0, 0, [0]).double().numpy()[0]
    n, tt = 0, 0.0
    while tt < budget_s and n < 64:
        t1 = time.perf_counter()
        oatt.paged_decode(q, kp, vp, perm.tolist(), L, wl.b, wl.scale)
        tt += time.perf_counter() - t1
        n += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": n * _kv_bytes(wl, [L]) / tt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": _cpu_model(),
            "sample": f"{n} decodes of one {L}-token sequence, layer 0 of {wl.name} (setup {time.perf_counter()-t0-tt:.1f}s untimed)"}


# ------------------------------------------------------------------ our arm

L2_FLUSH_DOC = ("L2 flushed before every timed step: a 256 MiB write, then a 256 MiB read of another buffer "
                "so that the write's dirty lines are written back before the step, not inside it")


class L2Flush:
    """Evicts L2 (129 MB) before a timed region: a 256 MiB write, then a read of another 256 MiB.
    The read pass leaves L2 holding clean lines of an unrelated buffer; without it, each miss of
    the timed kernel would first write back one dirty line of the flush, which charges the
    flush's own traffic to the kernel."""

    def __init__(self, dev, read_mib: int = 256):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(read_mib << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def _measure_device(wl, steps, warmup, dev, ws, kv="native", partition=0, fused=True, flush_l2=False,
                    min_seconds=0.0, auto_partition=False):
    """Time ``steps`` decode steps of ``wl`` on the device, inputs resident in HBM.

    The host plans of every step are made and uploaded first.  Without
    ``flush_l2`` the timed steps run back to back (for histories far larger than
    L2) and only the decode launches of the last timed steps are bracketed by
    events (an event between two launches ends their programmatic overlap).
    With ``flush_l2`` (histories that fit in L2) L2 is evicted before every
    timed step (``L2Flush``), each step is bracketed by its own events, and the
    step time is the sum of those.

    With ``min_seconds`` the ``steps`` planned steps are executed in turn as
    many times as it takes for the timed region to last about that long (sized
    by one untimed pass), so that the clock sampler sees the region; executing
    a planned step again repeats its copies, appends and decode exactly.
    Returns the Replay (for the e2e leg) and the figures of the run."""
    from paged_kv_cache_66_gb300 import api
    from paged_kv_cache_66_gb300.replay import Replay

    rp = Replay(wl, device=dev, kv=kv, partition_tokens=0 if auto_partition else (partition or None), fused=fused)
    rp.run_setup()
    torch.cuda.synchronize()
    total_steps = warmup + steps
    plans = [rp.plan_step(i) for i in range(total_steps)]
    dsteps = [rp.device_step(p) for p in plans]
    outs = [torch.empty((len(plans[0].uids), wl.Hq, wl.D), dtype=wl.torch_dtype, device=dev) for _ in rp.layers]
    flush = L2Flush(dev) if flush_l2 else None
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # The Python collector is left running: pausing it around the timed regions (gc.disable, with
    # or without a collection first) halved the host-bound one-layer config-2 step (~30 us of GPU
    # work per step).
    for i in range(warmup):
        rp.run_step(dsteps[i], outs)
    torch.cuda.synchronize()
    reps = 1
    if min_seconds > 0:
        t0 = time.perf_counter()
        for j in range(steps):
            if flush_l2:
                flush()
            rp.run_step(dsteps[warmup + j], outs)
        torch.cuda.synchronize()
        reps = max(1, int(np.ceil(min_seconds / max(time.perf_counter() - t0, 1e-6))))
    order = [warmup + n % steps for n in range(steps * reps)]
    planned_steps, steps = steps, steps * reps
    _barrier(ws)

    nL = len(rp.layers)
    # per-launch events on the decode launches of the last timed steps only (32 launches, or the
    # last quarter of the steps when fewer): bracketing every launch cost ~2.5 % of the
    # long-context step and ~30 % of the one-layer, L2-resident step
    ev_steps = steps if flush_l2 else min(max(1, -(-32 // nL)), max(1, steps // 4))
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(ev_steps * nL)]
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps if flush_l2 else 0)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    t_start.record(stream)
    for j in range(steps):
        ds = dsteps[order[j]]
        B, width = ds.tables.shape
        wsbuf = rp.workspace_for(B, width)
        if flush_l2:
            flush()
            ev_step[j][0].record(stream)
        torch.cuda.nvtx.range_push(f"decode step {j}")
        if ds.pairs.shape[0]:
            api.pa_copy_blocks(rp.k_pools, rp.v_pools, ds.pairs)
            launches += 1
        for li in range(nL):
            launches += rp.step_layer(li, outs[li], ds.q[li], ds.k_new[li], ds.v_new[li], ds.slots, ds.tables,
                                      ds.lens, wsbuf,
                                      events=ev_dec[(j - (steps - ev_steps)) * nL + li]
                                      if j >= steps - ev_steps else None, split=ds.splits[li])
            launches += 1 if wsbuf.numel() else 0
        torch.cuda.nvtx.range_pop()
        if flush_l2:
            ev_step[j][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    clk = clocks.stop()
    dev_ms = (sum(a.elapsed_time(b) for a, b in ev_step) if flush_l2 else t_start.elapsed_time(t_end))
    dev_ms_max = _max_over_ranks(dev_ms, ws, dev)
    timed = [dsteps[order[j]].plan for j in range(steps)]
    kv_bytes = sum(_kv_bytes(wl, p.lens, rp.kv_elt) for p in timed) * nL
    dec_ms = [a.elapsed_time(b) for a, b in ev_dec]
    dec_avg = sum(dec_ms) / len(dec_ms)
    alg = statistics.mean(_alg_bytes_decode(wl, p, rp.kv_elt, rp.fused) for p in timed[steps - ev_steps:])
    return rp, {
        "plans": plans, "nL": nL, "B": len(plans[0].uids), "dev_ms_max": dev_ms_max, "kv_bytes": kv_bytes,
        "steps": steps, "planned_steps": planned_steps,
        "launches": launches, "clocks": clk, "dec_avg_ms": dec_avg, "dec_med_ms": statistics.median(dec_ms),
        "alg": alg,
        "unique": statistics.mean(_unique_kv_bytes(wl, p, rp.kv_elt) for p in timed),
        "effective": statistics.mean(_kv_bytes(wl, p.lens, rp.kv_elt) for p in timed),
    }


# the other workloads' decode steps, measured in the same run after the headline
SECONDARY = [
    {"config": 4, "kv": "native"},
    {"config": 5, "combo": (128, 4, 16, "bf16"), "kv": "native"},
    {"config": 5, "combo": (256, 8, 16, "f16"), "kv": "native"},
    {"config": 5, "combo": (64, 8, 16, "bf16"), "kv": "native"},
    {"config": 5, "combo": (128, 8, 32, "bf16"), "kv": "native"},
    {"config": 2, "kv": "native"},
    # E4M3 pools take the library's automatic partition size (2048 tokens here): config 3 states
    # its 512-token split for 16-bit pools, where a token carries twice the bytes
    {"config": 3, "kv": "fp8", "auto_partition": True},
]
L2_BYTES = 129 << 20


def _history_bytes(wl, elt) -> int:
    """K/V bytes the setup writes (shared tokens once): the history one decode step reads."""
    tokens = sum(int(op[2]) for op in wl.setup_ops if op[0] == "write")
    return tokens * 2 * wl.Hkv * wl.D * elt * wl.layers


def _secondary(spec, steps, warmup, dev, ws, peak):
    """One entry of the ``configs`` record: a workload's decode step on its own clock record.
    A workload whose history is under 4x L2 is timed with L2 flushed before every step."""
    wl = _workload(spec["config"], warmup + steps + 1, spec.get("combo"))
    kv = spec["kv"]
    small = _history_bytes(wl, 1 if kv == "fp8" else wl.elt) < 4 * L2_BYTES
    auto = spec.get("auto_partition", False)
    rp, m = _measure_device(wl, steps, warmup, dev, ws, kv=kv, flush_l2=small, min_seconds=0.5,
                            auto_partition=auto)
    steps = m["steps"]
    ms = m["dev_ms_max"] / steps
    entry = {
        "workload": wl.name, "kv_cache": "e4m3" if kv == "fp8" else wl.dtype, "batch": m["B"],
        "partition_tokens": "automatic" if auto or not wl.partition_tokens else wl.partition_tokens,
        "layers": m["nL"], "steps": steps, "planned_steps": m["planned_steps"], "warmup": warmup,
        "ms_per_step": ms,
        "effective_kv_gbs": m["kv_bytes"] / (m["dev_ms_max"] / 1e3) / 1e9,
        "seq_steps_per_s": m["B"] * steps / (m["dev_ms_max"] / 1e3),
        "kv_bytes_per_decode": {"effective": m["effective"], "unique": m["unique"]},
        "l2": (L2_FLUSH_DOC + "; each step timed by its own events" if small
               else "history larger than L2 (no flush needed)"),
        "roofline": {"bound": "hbm", "peak": peak, "unit": "GB/s",
                     "alg_bytes_per_launch": m["alg"], "avg_launch_ms": m["dec_avg_ms"],
                     "median_launch_ms": m["dec_med_ms"],
                     "achieved": m["alg"] / (m["dec_avg_ms"] / 1e3) / 1e9,
                     "frac": m["alg"] / (m["dec_avg_ms"] / 1e3) / 1e9 / peak,
                     "unique_frac": m["unique"] / (m["dec_avg_ms"] / 1e3) / 1e9 / peak,
                     "step_frac": m["kv_bytes"] / (m["dev_ms_max"] / 1e3) / 1e9 / peak},
        "clocks": {k: m["clocks"][k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
        "gpu_launches": m["launches"],
    }
    if "combo" in spec:
        entry["combo"] = {"head_dim": wl.D, "group": wl.G, "block_size": wl.b, "dtype": wl.dtype}
    del rp
    torch.cuda.empty_cache()
    return entry


def run_ours(args, ws, rank, local):
    from paged_kv_cache_66_gb300 import api

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    api.pa_set_decode_kernel(args.kernel)
    api.pa_set_decode_heads_per_cta(args.heads_per_cta)
    total_steps = args.warmup + args.steps
    wl = _workload(args.config, total_steps + args.steps + 1, args.combo)
    if args.layers:
        wl.layers = min(wl.layers, args.layers)
    fp8_auto = args.kv == "fp8" and not args.partition  # E4M3 pools: the library's automatic size
    rp, m = _measure_device(wl, args.steps, args.warmup, dev, ws, kv=args.kv, partition=args.partition,
                            auto_partition=fp8_auto,
                            fused=not args.unfused, flush_l2=args.flush_l2)
    traffic = _profiled_traffic(_launch_key(args, wl, rp))
    plans, nL, B = m["plans"], m["nL"], m["B"]
    dev_ms_max = m["dev_ms_max"]
    kv_all = _sum_over_ranks(float(m["kv_bytes"]), ws, dev)
    value = kv_all / (dev_ms_max / 1e3) / 1e9
    seq_steps = B * args.steps * ws / (dev_ms_max / 1e3)
    dec_avg = m["dec_avg_ms"]
    peak, peak_kind = _peaks()
    achieved = m["alg"] / (dec_avg / 1e3) / 1e9
    err = api.pa_get_device_error()

    # ---------------- e2e through the public API with host buffers
    e2e = None if args.no_e2e else run_e2e(args, wl, rp, dev, ws)

    # ---------------- the other workloads (one GPU, headline workload only)
    configs = None
    if args.config == 3 and args.kv == "native" and not args.layers and not args.no_configs and ws == 1:
        del rp
        torch.cuda.empty_cache()
        configs = [_secondary(spec, 20, 3, dev, ws, peak) for spec in SECONDARY]
        err |= api.pa_get_device_error()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dev_ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype if args.kv == "native" else f"{wl.dtype}+e4m3-kv",
        "data": "synthetic",
        "config": {"workload": wl.name, "batch": B, "context": int(np.max(plans[0].lens)), "layers": nL,
                   "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.D, "block_size": wl.b,
                   "partition_tokens": ("automatic" if fp8_auto else
                                        wl.partition_tokens if not args.partition else args.partition),
                   "kv_cache": "e4m3" if args.kv == "fp8" else wl.dtype,
                   "l2": (L2_FLUSH_DOC + "; each step timed by its own events" if args.flush_l2
                          else "inputs larger than L2 (no flush needed)"),
                   "parallelism": f"replicas x{ws}"},
        "seq_steps_per_s": seq_steps,
        "kv_bytes_per_decode": {"effective": m["effective"], "unique": m["unique"],
                                "unique_gbs_per_launch": m["unique"] / (dec_avg / 1e3) / 1e9},
        "pct_hbm_peak": 100.0 * value / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": (f"pa_decode_append ({args.kernel} partition with the step's append + merge)"
                                if not args.unfused and args.kv == "native" and wl.dtype != "f32"
                                else f"pa_decode ({args.kernel} partition + merge)"),
                     "peak_kind": f"{peak_kind} hbm_gbs",
                     "alg_bytes_per_launch": m["alg"], "avg_launch_ms": dec_avg, "median_launch_ms": m["dec_med_ms"],
                     "launch_timing": ("avg_launch_ms is measured on event-bracketed launches of the last timed "
                                       "steps; ms_per_step on unbracketed steps, where consecutive launches "
                                       "overlap their ends, so layers x avg_launch_ms can exceed ms_per_step")},
        "clocks": {"sm_mhz": m["clocks"]["sm_mhz"], "sm_max_mhz": m["clocks"]["sm_max_mhz"],
                   "reasons": m["clocks"]["reasons"], "samples": m["clocks"]["samples"]},
        "e2e": e2e,
        "gpu_launches": m["launches"],
        "device_error_word": err,
    }
    if configs is not None:
        line["configs"] = configs
    if not args.no_cpu_baseline and ws == 1 and rank == 0:   # the host baseline: one GPU only
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line), flush=True)


def run_e2e(args, wl, rp, dev, ws):
    """K steps through the public API with host buffers (pinned), copies timed.

    Per step: the C++ plan writes slots / lengths / tables into one pinned
    metadata buffer (one host->device copy); the step's q, new K and new V rows
    of every layer are copied on the host into one pinned staging buffer (one
    host->device copy); every layer's output lands in one device buffer read
    back with one copy.  The pinned buffers form a small ring, each reused once
    its uploads are done, so the host works a few steps ahead of the device.
    """
    from paged_kv_cache_66_gb300 import api
    from workload import configs as wc
    # inputs of the next K steps, created on the host (not timed): positions
    # advance by one per step for this churn-free workload
    uids = list(wl.step_ops[rp.steps_done][-1][1])
    base = np.array([rp.host.length(u) for u in uids], dtype=np.int64)
    B, nL = len(uids), len(rp.layers)
    nq, nk = B * wl.Hq * wl.D, B * wl.Hkv * wl.D
    row = nq + 2 * nk
    host_in = []
    for j in range(args.steps):
        pos = base + j
        owners = np.array([wl.content_owner(u, int(p)) for u, p in zip(uids, pos)])
        x = torch.empty((nL, row), dtype=wl.torch_dtype)
        for li, layer in enumerate(rp.layers):
            x[li, :nq] = wc.q_rows(wl, layer, rp.steps_done + j, np.arange(B)).reshape(-1)
            x[li, nq:nq + nk] = wc.kv_rows(wl, layer, "k", owners, pos).reshape(-1)
            x[li, nq + nk:] = wc.kv_rows(wl, layer, "v", owners, pos).reshape(-1)
        host_in.append(x)
    stride = max(len(rp.host.table(u)) for u in uids) + args.steps // wl.b + 2
    meta_bytes = B * 8 + B * 4 + B * stride * 4

    def meta_views(buf):
        return (buf[:B * 8].view(torch.int64), buf[B * 8:B * 12].view(torch.int32),
                buf[B * 12:].view(torch.int32).view(B, stride))

    # a ring of pinned metadata buffers, each reused once its upload is done: the host may run up
    # to that many steps ahead of the device, so a host pause shorter than that costs nothing
    NMETA = 4
    bufs = [{"meta": torch.zeros(meta_bytes, dtype=torch.uint8).pin_memory(),
             "x": torch.empty((nL, row), dtype=wl.torch_dtype).pin_memory(), "ev": None} for _ in range(NMETA)]
    d_meta = torch.empty(meta_bytes, dtype=torch.uint8, device=dev)
    d_slots, d_lens, d_tables = meta_views(d_meta)
    d_x = torch.empty((nL, row), dtype=wl.torch_dtype, device=dev)
    d_q = [d_x[li, :nq].view(B, wl.Hq, wl.D) for li in range(nL)]
    d_k = [d_x[li, nq:nq + nk].view(B, wl.Hkv, wl.D) for li in range(nL)]
    d_v = [d_x[li, nq + nk:].view(B, wl.Hkv, wl.D) for li in range(nL)]
    d_out = torch.empty((nL, B, wl.Hq, wl.D), dtype=wl.torch_dtype, device=dev)
    out_host = torch.empty_like(d_out, device="cpu").pin_memory()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    _barrier(ws)
    h2d = d2h = 0
    kv = 0
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for j in range(args.steps):
        buf = bufs[j % NMETA]
        if buf["ev"] is not None:
            buf["ev"].synchronize()
        slots, lens, tables = meta_views(buf["meta"])
        ln = lens.numpy()
        pairs, width = rp.host.decode_step(uids, tables.numpy(), ln, slots.numpy())
        kv += _kv_bytes(wl, ln, rp.kv_elt) * nL
        d_meta.copy_(buf["meta"], non_blocking=True)
        h2d += meta_bytes
        if len(pairs):
            d_pairs = torch.as_tensor(pairs).pin_memory().to(dev, non_blocking=True)
            api.pa_copy_blocks(rp.k_pools, rp.v_pools, d_pairs)
            h2d += pairs.nbytes
        buf["x"].copy_(host_in[j])  # the step's inputs into pinned staging memory (host copy)
        d_x.copy_(buf["x"], non_blocking=True)
        buf["ev"] = torch.cuda.Event()
        buf["ev"].record(stream)  # both uploads from this ring slot are done past this point
        h2d += buf["x"].numel() * wl.elt
        wsbuf = rp.workspace_for(B, stride)
        for li in range(nL):
            rp.step_layer(li, d_out[li], d_q[li], d_k[li], d_v[li], d_slots, d_tables, d_lens, wsbuf)
        out_host.copy_(d_out, non_blocking=True)
        d2h += d_out.numel() * wl.elt
    t1.record(stream)
    torch.cuda.synchronize()
    rp.steps_done += args.steps
    ms = _max_over_ranks(t0.elapsed_time(t1), ws, dev)
    kv_all = _sum_over_ranks(float(kv), ws, dev)
    return {"value": kv_all / (ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d // args.steps,
            "d2h_bytes_per_step": d2h // args.steps, "ms_per_step": ms / args.steps}


def run_op(args, local):
    """Single-kernel measurements of the rows other than decode (not the default
    line): "append" = pa_kv_append of 8 x 4096 new tokens into a long-context
    pool; "copy" = pa_copy_blocks of 64 copy-on-write pairs over 32 layers;
    "host" = the C++ plan of one decode step (pa_host_decode_step) for the
    long-context and prefix-shared batches; "prefill" = pa_prefill of 8 chunks of
    1024 tokens over 3072 cached tokens each (Llama-3-8B-shaped layer)."""
    from paged_kv_cache_66_gb300 import api
    from paged_kv_cache_66_gb300.host import HostBlockManager
    peak, peak_kind = _peaks()
    K = max(args.steps, 5)
    if args.op != "host":
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K

    line = {"op": args.op, "n_gpus": 1, "steps": K, "warmup": args.warmup, "data": "synthetic"}
    if args.op == "append":
        N, Hkv, b, D = 20000, 8, 16, 128
        T = 8 * 4096
        kp = torch.zeros((N, Hkv, b, D), dtype=torch.float16, device=dev)
        vp = torch.zeros_like(kp)
        k = torch.randn((T, Hkv, D), device=dev).half()
        v = torch.randn((T, Hkv, D), device=dev).half()
        slots = (torch.randperm(N, device=dev)[: T // b].repeat_interleave(b) * b +
                 torch.arange(T, device=dev) % b).to(torch.int64)
        ms = timed(lambda: api.pa_kv_append(k, v, kp, vp, slots))
        alg = 2 * 2 * T * Hkv * D * 2 + 8 * T
        line.update(metric="pa_kv_append GB/s", value=alg / (ms / 1e3) / 1e9, unit="GB/s", ms_per_launch=ms,
                    config={"tokens": T, "kv_heads": Hkv, "head_dim": D, "block_size": b, "dtype": "f16"},
                    roofline={"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                              "frac": alg / (ms / 1e3) / 1e9 / peak, "alg_bytes_per_launch": alg,
                              "peak_kind": f"{peak_kind} hbm_gbs"})
    elif args.op == "copy":
        N, Hkv, b, D, L, n = 4096, 8, 16, 128, args.copy_layers, args.copy_pairs
        kps = [torch.randn((N, Hkv, b, D), device=dev).half() for _ in range(L)]
        vps = [torch.randn((N, Hkv, b, D), device=dev).half() for _ in range(L)]
        perm = torch.randperm(N, device=dev)
        pairs = torch.stack([perm[:n], perm[n:2 * n]], 1).to(torch.int64).contiguous()
        ms = timed(lambda: api.pa_copy_blocks(kps, vps, pairs))
        alg = n * L * 2 * 2 * Hkv * b * D * 2
        line.update(metric="pa_copy_blocks GB/s", value=alg / (ms / 1e3) / 1e9, unit="GB/s", ms_per_launch=ms,
                    config={"pairs": n, "layers": L, "block_bytes": Hkv * b * D * 2, "dtype": "f16"},
                    roofline={"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                              "frac": alg / (ms / 1e3) / 1e9 / peak, "alg_bytes_per_launch": alg,
                              "peak_kind": f"{peak_kind} hbm_gbs"})
    elif args.op == "prefill":
        wl = wcfg.prefill_config(dtype=args.prefill_dtype, head_dim=args.prefill_head_dim)
        kp, vp, q = wcfg.prefill_inputs(wl, device=dev)
        tables = torch.as_tensor(wl.tables(), device=dev)
        lens = torch.full((wl.batch,), wl.length, dtype=torch.int32, device=dev)
        qstart = torch.as_tensor(wl.qstart(), device=dev)
        out = torch.empty_like(q)
        flush = L2Flush(dev)  # before each launch
        for _ in range(args.warmup):
            api.pa_prefill(out, q, kp, vp, tables, lens, qstart, wl.scale, max_query_len=wl.chunk)
        torch.cuda.synchronize()
        # at least K launches, and enough for ~0.5 s so the clock sampler sees the region (a
        # dense kernel on this part may run under its power cap: the clocks say)
        t0 = time.perf_counter()
        flush()
        api.pa_prefill(out, q, kp, vp, tables, lens, qstart, wl.scale, max_query_len=wl.chunk)
        torch.cuda.synchronize()
        K = max(K, int(np.ceil(0.5 / max(time.perf_counter() - t0, 1e-6))))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        clocks = ClockSampler(local)
        for a, b_ in ev:
            flush()
            a.record(stream)
            api.pa_prefill(out, q, kp, vp, tables, lens, qstart, wl.scale, max_query_len=wl.chunk)
            b_.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
        ms = sum(a.elapsed_time(b_) for a, b_ in ev) / K
        line["steps"] = K
        flops = 4 * wl.D * wl.Hq * wl.causal_pairs()
        tf = flops / (ms / 1e3) / 1e12
        tpeak, tkind = _tensor_peak()
        line.update(metric="pa_prefill TFLOP/s (causal pairs x 4 D x Hq)", value=tf, unit="TFLOP/s",
                    ms_per_launch=ms, dtype=wl.dtype,
                    config={"workload": wl.name, "batch": wl.batch, "history": wl.history, "chunk": wl.chunk,
                            "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.D, "block_size": wl.b,
                            "l2": L2_FLUSH_DOC.replace("step", "launch")},
                    tokens_per_s=wl.batch * wl.chunk / (ms / 1e3),
                    roofline={"bound": "tensor", "achieved": tf, "peak": tpeak, "unit": "TFLOP/s", "frac": tf / tpeak,
                              "alg_flops_per_launch": flops, "peak_kind": tkind, "traffic": None,
                              "kernel": "pa_prefill (tcgen05, persistent CTAs, 128-key tiles)" if wl.D <= 128
                              else "pa_prefill (tcgen05, Q in tensor memory)"},
                    clocks={k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
                    gpu_launches=K)
    else:
        res = {}
        for name, wl in (("longctx-f16-b8x32k", wcfg.config3(steps=K + args.warmup, layers=1)),
                         ("prefix-shared-bf16-b256", wcfg.config4(steps=K + args.warmup))):
            h = HostBlockManager(wl.num_blocks, wl.b, wl.free_order)
            for op in wl.setup_ops:           # host state only (no device writes)
                if op[0] == "create":
                    h.create(op[1])
                elif op[0] == "write":
                    h.reserve(op[1], op[2])
                    h.advance(op[1], op[2])
                elif op[0] == "fork":
                    h.fork(op[1], op[2])
                elif op[0] == "truncate":
                    h.truncate(op[1], op[2])
            uids = list(wl.step_ops[0][-1][1])
            B = len(uids)
            stride = max(len(h.table(u)) for u in uids) + K + args.warmup + 2
            tables = np.zeros((B, stride), np.int32)
            lens = np.zeros(B, np.int32)
            slots = np.zeros(B, np.int64)
            for _ in range(args.warmup):
                h.decode_step(uids, tables, lens, slots)
            t0 = time.perf_counter()
            for _ in range(K):
                h.decode_step(uids, tables, lens, slots)
            res[name] = {"batch": B, "us_per_step": 1e6 * (time.perf_counter() - t0) / K}
        line.update(metric="host decode-step plan us", value=res["longctx-f16-b8x32k"]["us_per_step"], unit="us",
                    higher_is_better=False, config=res)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--combo", type=str, default="128,4,16,bf16", help="config 5: D,G,b,dtype")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' record")
    ap.add_argument("--flush-l2", action="store_true",
                    help="evict L2 before every timed step (for workloads whose history fits in L2)")
    ap.add_argument("--layers", type=int, default=0, help="use the first N layers only (profiling)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "mma"], help="decode partition kernel")
    ap.add_argument("--heads-per-cta", type=int, default=0, choices=[0, 1, 2],
                    help="tensor-core decode: KV heads per CTA (0: chosen per launch)")
    ap.add_argument("--unfused", action="store_true",
                    help="decode step: separate append and decode launches instead of pa_decode_append")
    ap.add_argument("--kv", default="native", choices=["native", "fp8"], help="KV cache storage (fp8 = E4M3)")
    ap.add_argument("--partition", type=int, default=0, help="decode partition tokens (0: the workload's)")
    ap.add_argument("--copy-layers", type=int, default=32, help="--op copy: layers (pools of 4096 blocks each)")
    ap.add_argument("--copy-pairs", type=int, default=64, help="--op copy: copy-on-write pairs")
    ap.add_argument("--prefill-head-dim", type=int, default=128, choices=[64, 128, 256],
                    help="--op prefill head dim (Hq 32, Hkv 8 kept)")
    ap.add_argument("--prefill-dtype", default="bf16", choices=["f16", "bf16"], help="--op prefill storage dtype")
    ap.add_argument("--op", default="step", choices=["step", "append", "copy", "host", "prefill"],
                    help="step = the benchmark line; others measure one row of the path alone")
    args = ap.parse_args()
    D, G, b, dt = args.combo.split(",")
    args.combo = (int(D), int(G), int(b), dt)
    if args.warmup < 3:
        raise SystemExit("warmup must be >= 3")
    ws, rank, local = _dist()
    if args.op != "step":
        run_op(args, local)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
