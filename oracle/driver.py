"""Replay a ``workload`` op list through the oracle's block manager and pools.

For every op the oracle records what the device must be given (copy pairs,
slots, block tables, lengths); with ``pools=True`` it also keeps its own K/V
pools (``cache_ops``) so the whole pool state can be compared bit for bit, and
attention gathers through its own tables.  With ``pools=False`` (workloads too
large to mirror on the host) attention is computed from the token contents the
workload defines for each position, which checks the table, append and
copy-on-write chain end to end.

One decode step ([P1] "The paged cache", flow per step; [P4] "Block table and
allocator", decode step): reserve one position per sequence (copy-on-write
decisions in batch order), copy the recorded block pairs in every layer,
append the new K/V row of every sequence at its old length, commit the
lengths, then attend with one query per sequence over the new length.
"""
from __future__ import annotations

import numpy as np

from workload import configs as wcfg

from . import attention, cache_ops, quant
from .blocks import SeqTables


class OracleRun:
    def __init__(self, wl, pools: bool = True, layers=None, kv: str = "native", input_device="cpu"):
        """kv = "fp8": the K/V history is what E4M3 pools with the workload's
        per-(layer, KV head) scales store (content route only).

        input_device: where the seeded generator (``workload``) draws the q and
        K/V values of the content route before they come to the host.  The
        generator is bit-identical on every device, and all of the oracle's
        arithmetic runs here in fp64 whatever the choice; a device only makes
        drawing the long histories of the large workloads fast."""
        self.kv = kv
        self.input_device = input_device
        if kv == "fp8" and pools:
            raise ValueError("the FP8 replay uses the content route (pools=False)")
        self.wl = wl
        self.t = SeqTables(wl.num_blocks, wl.b, wl.free_order)
        self.layers = list(range(wl.layers)) if layers is None else list(layers)
        self.pools = pools
        self.k_pool, self.v_pool = {}, {}
        if pools:
            for layer in self.layers:
                self.k_pool[layer] = cache_ops.new_pool(wl.num_blocks, wl.Hkv, wl.b, wl.D,
                                                        wl.torch_dtype)
                self.v_pool[layer] = cache_ops.new_pool(wl.num_blocks, wl.Hkv, wl.b, wl.D,
                                                        wl.torch_dtype)
        self.steps_done = 0

    # ------------------------------------------------------------------ writes
    def _write_rows(self, uids, positions, slots, pairs):
        if not self.pools:
            return
        wl = self.wl
        cache_ops.copy_blocks([self.k_pool[x] for x in self.layers],
                              [self.v_pool[x] for x in self.layers], pairs)
        owners = [wl.content_owner(u, p) for u, p in zip(uids, positions)]
        for layer in self.layers:
            k = wcfg.kv_rows(wl, layer, "k", owners, positions)
            v = wcfg.kv_rows(wl, layer, "v", owners, positions)
            cache_ops.append(self.k_pool[layer], self.v_pool[layer], k, v, slots, wl.b)

    def apply(self, op) -> dict:
        kind = op[0]
        t = self.t
        rec = {"op": kind}
        if kind == "create":
            t.create(op[1])
        elif kind == "write":
            uid, n = op[1], int(op[2])
            start = t.lengths[uid]
            pairs = t.reserve(uid, n)
            positions = list(range(start, start + n))
            slots = [t.slot(uid, p) for p in positions]
            self._write_rows([uid] * n, positions, slots, pairs)
            t.advance(uid, n)
            rec.update(uid=uid, pairs=pairs, slots=slots, positions=positions)
        elif kind == "fork":
            t.fork(op[1], op[2])
        elif kind == "truncate":
            t.truncate(op[1], op[2])
        elif kind == "free":
            t.free(op[1])
        elif kind == "step":
            uids = list(op[1])
            pairs = []
            for u in uids:
                pairs += t.reserve(u, 1)
            positions = [t.lengths[u] for u in uids]
            slots = [t.slot(u, p) for u, p in zip(uids, positions)]
            self._write_rows(uids, positions, slots, pairs)
            for u in uids:
                t.advance(u, 1)
            tables, lens = t.batch(uids)
            rec.update(uids=uids, pairs=pairs, slots=slots, positions=positions,
                       tables=tables, lens=lens, step=self.steps_done)
            self.steps_done += 1
        else:
            raise ValueError(f"unknown op {kind}")
        return rec

    def run_setup(self):
        return [self.apply(op) for op in self.wl.setup_ops]

    def run_step_ops(self, step_index: int):
        return [self.apply(op) for op in self.wl.step_ops[step_index]]

    # --------------------------------------------------------------- attention
    def attend(self, rec: dict, layer: int, rows=None) -> np.ndarray:
        """fp64 outputs [len(rows), Hq, D] for batch rows of a recorded step."""
        wl = self.wl
        rows = list(range(len(rec["uids"]))) if rows is None else list(rows)
        q = wcfg.q_rows(wl, layer, rec["step"], rows, device=self.input_device).cpu().double().numpy()
        out = np.zeros((len(rows), wl.Hq, wl.D), dtype=np.float64)
        for i, r in enumerate(rows):
            L = int(rec["lens"][r])
            if self.pools:
                out[i] = attention.paged_decode(q[i], self.k_pool[layer], self.v_pool[layer],
                                                rec["tables"][r], L, wl.b, wl.scale)
            else:
                K, V = self.history(rec["uids"][r], L, layer)
                out[i] = attention.decode_attention(q[i], K, V, wl.scale)
        return out

    def history(self, uid, length: int, layer: int):
        """Contiguous fp64 K, V [L, Hkv, D] from the workload's token contents."""
        wl = self.wl
        pos = np.arange(length, dtype=np.int64)
        owners = wl.content_owners(uid, pos)
        K = wcfg.kv_rows(wl, layer, "k", owners, pos, device=self.input_device).cpu()
        V = wcfg.kv_rows(wl, layer, "v", owners, pos, device=self.input_device).cpu()
        if self.kv == "fp8":
            ks, vs = wcfg.kv_scales(wl, layer, "k"), wcfg.kv_scales(wl, layer, "v")
            K = quant.dequantize(quant.quantize_rows(K.float().numpy(), ks), ks, head_axis=1)
            V = quant.dequantize(quant.quantize_rows(V.float().numpy(), vs), vs, head_axis=1)
            return K, V
        return K.double().numpy(), V.double().numpy()
