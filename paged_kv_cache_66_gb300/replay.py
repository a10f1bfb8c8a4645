"""Drive a seeded workload through the host block manager and the kernels.

One decode step ("25. Paged attention and prefix caching", section "The paged
cache", flow per step):
  0. host: frees and arrivals of the step; an arrival's prompt write is
     reserved and given its slots
  1. host: reserve one position per sequence (copy-on-write pairs), slot of
     the new position, length + 1, padded block tables   (C++ manager)
  2. device: one pa_copy_blocks over every layer for all the step's pairs
  3. device, per layer: the step's new K/V rows into the pool, then the
     decode: pa_kv_append of the arrivals' prompt rows and one pa_decode_append
     that writes each sequence's newest row and decodes (16-bit pools), or one
     pa_kv_append of all the rows followed by pa_decode
The host part of a step is planned separately (``plan_step``) from its device
part (``run_step``) so that a benchmark can keep the plans of many steps
resident on the device and time the device path alone.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from workload import configs as wcfg

from . import api
from .host import HostBlockManager


@dataclass
class PendingWrite:
    """A prompt write planned on the host, executed on the device with its step."""
    pairs: np.ndarray          # [n, 2] int64 copy-on-write pairs
    slots: np.ndarray          # [T] int64
    owners: np.ndarray         # [T] content owner of each position
    positions: np.ndarray      # [T] int64


@dataclass
class StepPlan:
    step: int
    uids: list
    slots: np.ndarray          # [B] int64
    pairs: np.ndarray          # [n, 2] int64
    tables: np.ndarray         # [B, width] int32
    lens: np.ndarray           # [B] int32
    positions: np.ndarray      # [B] int64 (position of the appended token)
    writes: list = None        # prompt writes of arrivals, run before the decode step


@dataclass
class DeviceStep:
    """A step's metadata and inputs, resident on the device (appends and copies of
    the whole step, arrivals' prompts included)."""
    plan: StepPlan
    slots: torch.Tensor
    pairs: torch.Tensor
    tables: torch.Tensor
    lens: torch.Tensor
    q: list                    # per layer [B, Hq, D]
    k_new: list                # per layer [T, Hkv, D]: arrivals' prompt rows, then one row per sequence
    v_new: list
    splits: list = None        # per layer: the rows split into arrivals and newest rows (views, made once)


class Replay:
    def __init__(self, wl, device="cuda", layers=None, partition_tokens=None, kv="native", fused=True,
                 gen_device=None):
        """kv = "native": pools in the workload's dtype; kv = "fp8": E4M3 pools
        with the workload's per-(layer, KV head) scales.  fused: each layer's
        newest rows go with its decode in one pa_decode_append (16-bit pools).
        gen_device: where the seeded generator draws q and the new K/V rows
        (default: the pools' device); drawn elsewhere, each tensor is moved to
        the pools' device in one copy."""
        self.wl = wl
        self.fused = fused and kv == "native" and wl.dtype in ("f16", "bf16")
        self.device = torch.device(device)
        self.gen_device = self.device if gen_device is None else torch.device(gen_device)
        self.layers = list(range(wl.layers)) if layers is None else list(layers)
        self.host = HostBlockManager(wl.num_blocks, wl.b, wl.free_order)
        self.kv = kv
        shape = (wl.num_blocks, wl.Hkv, wl.b, wl.D)
        pool_dtype = torch.uint8 if kv == "fp8" else wl.torch_dtype
        self.k_pools = [torch.zeros(shape, dtype=pool_dtype, device=self.device) for _ in self.layers]
        self.v_pools = [torch.zeros(shape, dtype=pool_dtype, device=self.device) for _ in self.layers]
        if kv == "fp8":
            self.k_scales = [torch.as_tensor(wcfg.kv_scales(wl, layer, "k")).to(self.device) for layer in self.layers]
            self.v_scales = [torch.as_tensor(wcfg.kv_scales(wl, layer, "v")).to(self.device) for layer in self.layers]
        self.partition_tokens = wl.partition_tokens if partition_tokens is None else partition_tokens
        self.steps_done = 0
        self._ws = torch.empty(0, dtype=torch.uint8, device=self.device)

    @property
    def kv_elt(self) -> int:
        """Bytes per stored K/V element."""
        return 1 if self.kv == "fp8" else self.wl.elt

    def append(self, li: int, k, v, slots, stream=None):
        """pa_kv_append (or its FP8 form) into layer slot li."""
        if self.kv == "fp8":
            api.pa_kv_append_fp8(k, v, self.k_pools[li], self.v_pools[li], self.k_scales[li], self.v_scales[li],
                                 slots, stream=stream)
        else:
            api.pa_kv_append(k, v, self.k_pools[li], self.v_pools[li], slots, stream=stream)

    def decode(self, li: int, out, q, tables, lens, workspace, stream=None):
        """pa_decode (or its FP8 form) over layer slot li."""
        ws = workspace if workspace is not None and workspace.numel() else None
        if self.kv == "fp8":
            api.pa_decode_fp8(out, q, self.k_pools[li], self.v_pools[li], self.k_scales[li], self.v_scales[li],
                              tables, lens, self.wl.scale, partition_tokens=self.partition_tokens, workspace=ws,
                              stream=stream)
        else:
            api.pa_decode(out, q, self.k_pools[li], self.v_pools[li], tables, lens, self.wl.scale,
                          partition_tokens=self.partition_tokens, workspace=ws, stream=stream)

    @staticmethod
    def split_rows(B: int, k_new, v_new, slots):
        """(arrivals' K, V, slots, newest rows' K, V, slots): views of the step's rows, the
        arrivals' part None when there are none.  Made once per step outside any timed loop
        (each view costs the host a few microseconds)."""
        T = k_new.shape[0]
        if T == B:
            return None, None, None, k_new, v_new, slots
        return k_new[:T - B], v_new[:T - B], slots[:T - B], k_new[T - B:], v_new[T - B:], slots[T - B:]

    def step_layer(self, li: int, out, q, k_new, v_new, slots, tables, lens, workspace, stream=None,
                   events=None, split=None) -> int:
        """One layer of a decode step: the step's rows into the pool, then the
        decode.  k_new / v_new / slots hold the arrivals' prompt rows first, then
        one row per sequence (its newest position); with `fused` those last B rows
        go with the decode in one pa_decode_append (`split`: split_rows of them, if
        already made).  `events` (a pair) brackets the decode launch.  Returns the
        number of launches made (merge not counted)."""
        launches = 0
        if not self.fused:
            self.append(li, k_new, v_new, slots, stream=stream)
            launches += 1
        else:
            k_arr, v_arr, s_arr, k_last, v_last, s_last = (split if split is not None else
                                                           self.split_rows(q.shape[0], k_new, v_new, slots))
            if k_arr is not None:
                self.append(li, k_arr, v_arr, s_arr, stream=stream)
                launches += 1
        if events is not None:
            events[0].record(stream if stream is not None else torch.cuda.current_stream())
        if self.fused:
            ws = workspace if workspace is not None and workspace.numel() else None
            api.pa_decode_append(out, q, k_last, v_last, s_last, self.k_pools[li],
                                 self.v_pools[li], tables, lens, self.wl.scale, partition_tokens=self.partition_tokens,
                                 workspace=ws, stream=stream)
        else:
            self.decode(li, out, q, tables, lens, workspace, stream=stream)
        if events is not None:
            events[1].record(stream if stream is not None else torch.cuda.current_stream())
        return launches + 1

    # ------------------------------------------------------------------ ops
    def _copy(self, pairs: np.ndarray):
        if len(pairs):
            p = torch.as_tensor(np.asarray(pairs, dtype=np.int64).reshape(-1, 2)).to(self.device)
            api.pa_copy_blocks(self.k_pools, self.v_pools, p)

    def _write_host(self, uid: int, n: int) -> "PendingWrite":
        """Host part of a prompt write: reserve, slots, commit the length."""
        start = self.host.length(uid)
        pairs = np.array(self.host.reserve(uid, n), dtype=np.int64).reshape(-1, 2)
        slots = self.host.slots(uid, start, n)
        pos = np.arange(start, start + n, dtype=np.int64)
        self.host.advance(uid, n)
        return PendingWrite(pairs, slots, self.wl.content_owners(uid, pos), pos)

    def _write_device(self, w: "PendingWrite", stream=None):
        """Device part: copy-on-write copies, then the K/V rows of every layer."""
        wl = self.wl
        if len(w.pairs):
            api.pa_copy_blocks(self.k_pools, self.v_pools, torch.as_tensor(w.pairs).to(self.device), stream=stream)
        slots_d = torch.as_tensor(w.slots).to(self.device)
        n = len(w.slots)
        chunk = 1 << 14
        for li, layer in enumerate(self.layers):
            for c0 in range(0, n, chunk):
                c1 = min(n, c0 + chunk)
                k = wcfg.kv_rows(wl, layer, "k", w.owners[c0:c1], w.positions[c0:c1],
                                 device=self.gen_device).to(self.device)
                v = wcfg.kv_rows(wl, layer, "v", w.owners[c0:c1], w.positions[c0:c1],
                                 device=self.gen_device).to(self.device)
                self.append(li, k, v, slots_d[c0:c1], stream=stream)

    def _write(self, uid: int, n: int):
        self._write_device(self._write_host(uid, n))

    def apply(self, op):
        kind = op[0]
        h = self.host
        if kind == "create":
            h.create(op[1])
        elif kind == "write":
            self._write(op[1], int(op[2]))
        elif kind == "fork":
            h.fork(op[1], op[2])
        elif kind == "truncate":
            h.truncate(op[1], op[2])
        elif kind == "free":
            h.free(op[1])
        else:
            raise ValueError(f"op {kind} is not a setup op")

    def run_setup(self):
        for op in self.wl.setup_ops:
            self.apply(op)

    # ------------------------------------------------------------------ steps
    def plan_step(self, step_index: int) -> StepPlan:
        """Host part of one step: the step's frees and arrivals (their prompt
        writes are planned, not yet executed), then the decode step itself."""
        ops = self.wl.step_ops[step_index]
        plan = None
        writes = []
        for op in ops:
            if op[0] == "write":
                writes.append(self._write_host(op[1], int(op[2])))
                continue
            if op[0] != "step":
                self.apply(op)
                continue
            uids = list(op[1])
            B = len(uids)
            positions = np.array([self.host.length(u) for u in uids], dtype=np.int64)
            stride = max(len(self.host.table(u)) for u in uids) + 1
            tables = np.zeros((B, stride), dtype=np.int32)
            lens = np.zeros(B, dtype=np.int32)
            slots = np.zeros(B, dtype=np.int64)
            pairs, w = self.host.decode_step(uids, tables, lens, slots)
            plan = StepPlan(self.steps_done, uids, slots, pairs, np.ascontiguousarray(tables[:, :w]), lens,
                            positions, writes)
            self.steps_done += 1
        return plan

    def device_step(self, plan: StepPlan) -> DeviceStep:
        """Upload the plan and generate the step's q and new K/V rows on the device.

        Every row the step appends -- the prompts of arriving sequences, then one
        token per decoding sequence in batch order -- is generated per layer
        (step_layer writes them), and every copy-on-write pair goes into one
        pa_copy_blocks (copies first: a copy's source is a shared block, which no
        append of the step touches)."""
        wl, dev = self.wl, self.device
        writes = plan.writes or []
        owners = np.array([wl.content_owner(u, int(p)) for u, p in zip(plan.uids, plan.positions)])
        all_owners = np.concatenate([w.owners for w in writes] + [owners])
        all_pos = np.concatenate([w.positions for w in writes] + [plan.positions])
        all_slots = np.concatenate([w.slots for w in writes] + [plan.slots])
        all_pairs = np.concatenate([w.pairs.reshape(-1, 2) for w in writes] + [plan.pairs.reshape(-1, 2)])
        rows = np.arange(len(plan.uids))
        q, kn, vn = [], [], []
        gd = self.gen_device
        for layer in self.layers:
            q.append(wcfg.q_rows(wl, layer, plan.step, rows, device=gd).to(dev))
            kn.append(wcfg.kv_rows(wl, layer, "k", all_owners, all_pos, device=gd).to(dev))
            vn.append(wcfg.kv_rows(wl, layer, "v", all_owners, all_pos, device=gd).to(dev))
        d_slots = torch.as_tensor(all_slots).to(dev)
        B = len(plan.uids)
        splits = [self.split_rows(B, k, v, d_slots) for k, v in zip(kn, vn)]
        return DeviceStep(plan, d_slots, torch.as_tensor(all_pairs).to(dev),
                          torch.as_tensor(plan.tables).to(dev), torch.as_tensor(plan.lens).to(dev), q, kn, vn, splits)

    def workspace_for(self, batch: int, max_blocks: int) -> torch.Tensor:
        wl = self.wl
        need = api.pa_decode_workspace_size(batch, wl.Hq, wl.D, max_blocks, wl.b, self.partition_tokens)
        if self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def run_step(self, ds: DeviceStep, outs=None, stream=None) -> list:
        """Device part of one decode step over every layer; returns outputs."""
        wl = self.wl
        B, width = ds.tables.shape
        ws = self.workspace_for(B, width)
        # one NVTX range per step and per layer (free unless a profiler listens)
        torch.cuda.nvtx.range_push(f"step {ds.plan.step}")
        if ds.pairs.shape[0]:
            api.pa_copy_blocks(self.k_pools, self.v_pools, ds.pairs, stream=stream)
        if outs is None:
            outs = [torch.empty((B, wl.Hq, wl.D), dtype=wl.torch_dtype, device=self.device) for _ in self.layers]
        for li in range(len(self.layers)):
            torch.cuda.nvtx.range_push(f"layer {self.layers[li]}")
            self.step_layer(li, outs[li], ds.q[li], ds.k_new[li], ds.v_new[li], ds.slots, ds.tables, ds.lens, ws,
                            stream=stream, split=ds.splits[li] if ds.splits else None)
            torch.cuda.nvtx.range_pop()
        torch.cuda.nvtx.range_pop()
        return outs
