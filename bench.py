#!/usr/bin/env python
"""Benchmark of the kvattn hot path on GB300: one step = the host block
allocator, RoPE + KV-cache append of the step's new tokens, chunked-prefill
attention (mixed workload) and split-KV decode attention, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5|c4|c3|c2|c1]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

Prints ONE JSON line (rank 0).  `value` is KV bytes read by the step's
attention kernels / device step time with every input resident in HBM
(whole job over N GPUs); `e2e` is the same metric through the C ABI from
pinned host buffers, with the host<->device copies inside the timed region.
For N > 1 (torchrun) each rank runs its own replica of the workload on its
own GPU (the path shards by sequence; no collective in the data path).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode attention KV-read GB/s and % of GB300 HBM peak; query tokens/s"
DEFAULT_WORKLOAD = "c5"   # the only workload whose step runs every stage: allocator, rope_append, prefill, decode


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default=DEFAULT_WORKLOAD)
    p.add_argument("--rows", type=int, default=0,
                   help="use only the first N decode rows of the workload (profiling small cases)")
    p.add_argument("--chunks", type=int, default=-1,
                   help="use only the first N prefill chunks of the workload (profiling small cases)")
    p.add_argument("--compact-pool", action="store_true",
                   help="pool of twice the blocks the batch needs instead of the workload's pool size")
    p.add_argument("--layers", type=int, default=1,
                   help="run the step over L layers: one multi-layer cache, each layer's q/k/v taken as views "
                        "of its own fused QKV projection output, rotated q into a dense buffer")
    p.add_argument("--kv-dtype", choices=["model", "fp8"], default="model",
                   help="fp8: e4m3 KV cache with a scale per (slot, head) (bf16 workloads, head_dim 128)")
    p.add_argument("--graph", action="store_true",
                   help="also time launch-bound small workloads as CUDA-graph replays of 50 steps (L2 warm) "
                        "and as single steps after an L2 flush")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the per-config lines (decode-only configs, launch-bound graphs, 32 layers) that "
                        "the default run adds after the headline workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1898.0)), float(
            d.get("bf16_tflops_sustained", 1718.7)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- multi-rank

def max_over_ranks(values, device=None):
    """Element-wise max of per-rank floats over the process group (identity
    when torch.distributed is not initialised): the job takes as long as its
    slowest rank."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, max_elapsed_s: float) -> float:
    """Units all ranks processed per second (weak scaling: every rank runs a replica)."""
    return world * steps * units_per_rank_step / max_elapsed_s


# ----------------------------------------------------------------------------- ncu traffic

KERNEL_SOURCES = {"decode_split+decode_combine": "decode.cu", "prefill_chunk": "prefill.cu",
                  "rope_append": "rope_append.cu"}


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) of `kernel` on `workload` from the
    committed ncu summary, or None when it was taken on other source code."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = KERNEL_SOURCES.get(kernel)
    if not src or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel, {}).get(workload)
    if not rec:
        return None
    with open(os.path.join(ROOT, "kv_cache_attention_rope_gb300", "csrc", src), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    return rec["bytes_per_launch"] if rec.get("source_sha256") == sha else None


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import torch

        try:
            self.idx = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.idx = str(device.index)
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- our arm

class Step:
    """A workload's step on one GPU, inputs resident in HBM."""

    def __init__(self, wl: workloads.Workload, device, rows: int = 0, compact_pool: bool = False, chunks: int = -1,
                 layers: int = 1, kv_fp8: bool = False):
        import torch

        import kv_cache_attention_rope_gb300 as kv

        self.kv, self.torch, self.wl, self.dev = kv, torch, wl, device
        self.layers = max(1, int(layers))
        self.fp8 = bool(kv_fp8)
        dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.dt = dt
        H, D, BS = wl.num_kv_heads, wl.head_dim, wl.block_size
        per_block = 2 * BS * H * D * wl.elem_bytes
        if self.fp8:
            per_block = 2 * BS * H * (D + 4)   # e4m3 codes + one fp32 scale per (slot, head), K and V
        nb = None
        subset = None
        if rows or chunks >= 0:
            nc = wl.chunks if chunks < 0 else min(chunks, wl.chunks)
            nd = wl.decode_batch if not rows else min(rows, wl.decode_batch)
            if nc != wl.chunks:
                wl = dataclasses.replace(wl, chunks=nc)
                self.wl = wl
            subset = list(range(nc)) + list(range(nc, nc + nd))
        if self.fp8 and (wl.dtype != "bf16" or wl.head_dim != 128 or self.layers > 1):
            raise SystemExit("--kv-dtype fp8: bf16 workloads with head_dim 128, one layer")
        if wl.layout == "paged":
            if compact_pool:
                probe = workloads.make_batch(wl, num_blocks=1 << 30, rows_subset=subset)
                nb = int(2 * ((probe.total + BS - 1) // BS).sum())
            elif wl.pool_bytes:
                nb = wl.pool_bytes // per_block
        self.cfg = kv.make_config(wl.num_q_heads, H, D, kv.BF16 if wl.dtype == "bf16" else kv.F32)
        # batch (prefill chunks first, then decode rows); shrink a huge pool until it fits
        while True:
            batch = workloads.make_batch(wl, num_blocks=nb, rows_subset=subset)
            try:
                if self.fp8:
                    self.caches = [kv.CacheFP8.empty(batch.num_blocks, H, BS, device)]
                elif self.layers == 1:
                    self.caches = [kv.Cache.empty(batch.num_blocks, H, BS, D, dt, device)]
                else:
                    # one block id names 2 x layers regions of one allocation
                    self.layered = kv.LayeredCache.empty(self.cfg, self.layers, batch.num_blocks, BS, dt, device)
                    self.caches = [self.layered.layer(l) for l in range(self.layers)]
                break
            except torch.OutOfMemoryError:
                nb = batch.num_blocks // 2
                torch.cuda.empty_cache()
        cache = self.caches[0]
        self.batch, self.cache = batch, cache
        self.pool_bytes = batch.num_blocks * per_block * self.layers
        nchunk = wl.chunks
        self.nchunk = nchunk
        past, new = batch.past, batch.new
        # ---- host block allocator adopts the table; blocks opened by this step's
        # tokens are handed out by the allocator every step and returned after it
        self.alloc = kv.BlockAllocator(batch.num_blocks)
        self.table_host = batch.block_table.copy()
        self.open_cells = []
        if wl.layout == "paged":
            for r in range(batch.rows):
                first_new_block = (int(past[r]) + BS - 1) // BS
                last_block = (int(past[r] + new[r]) - 1) // BS
                for c in range(first_new_block, last_block + 1):
                    self.open_cells.append((r, c))
            rr = np.array([r for r, _ in self.open_cells], dtype=np.int64)
            cc = np.array([c for _, c in self.open_cells], dtype=np.int64)
            self.open_r, self.open_c = rr, cc
            self.table_host[rr, cc] = -1
            self.alloc.claim(self.table_host[self.table_host >= 0])
            ids = self.alloc.alloc(len(rr))
            self.table_host[rr, cc] = ids
            self.alloc.free(ids[::-1])      # LIFO: the next step gets the same ids in the same order
            self.step_ids = ids
        self.d_table = torch.from_numpy(self.table_host).to(device)
        # ---- cache history (positions 0..past-1) drawn on the device
        gen = torch.Generator(device=device)
        gen.manual_seed(workloads.DATA_SEED)
        rows = np.repeat(np.arange(batch.rows), past)
        pos = np.concatenate([np.arange(p) for p in past]) if past.sum() else np.zeros(0, np.int64)
        blk = self.table_host[rows, pos // BS].astype(np.int64)
        off = (pos % BS).astype(np.int64)
        step = 1 << 17
        if self.fp8:
            # every page of a block holding history: finite e4m3 codes of both signs, positive scales
            used = torch.from_numpy(np.unique(blk)).to(device)
            pool = self.caches[0].pool
            for s0 in range(0, len(used), 1 << 14):
                ids = used[s0:s0 + (1 << 14)]
                shp = (len(ids),) + tuple(pool.shape[1:3])
                codes = torch.randint(0, 0x7F, shp + (4096,), generator=gen, device=device, dtype=torch.uint8)
                sign = torch.randint(0, 2, shp + (4096,), generator=gen, device=device, dtype=torch.uint8)
                scales = torch.rand(shp + (32,), generator=gen, device=device) * 0.02 + 0.001
                pool[ids] = torch.cat([codes | (sign << 7), scales.view(torch.uint8)], dim=3)
        for c in ([] if self.fp8 else self.caches):
            for s in range(0, len(pos), step):
                b = torch.from_numpy(blk[s:s + step]).to(device)
                o = torch.from_numpy(off[s:s + step]).to(device)
                n = len(b)
                c.k_pool[b, :, o, :] = torch.randn((n, H, D), generator=gen, device=device).to(dt)
                c.v_pool[b, :, o, :] = torch.randn((n, H, D), generator=gen, device=device).to(dt)
        # ---- this step's new tokens (prefill chunk tokens, then one per decode row)
        q_l, k_l, v_l, p_l, s_l = [], [], [], [], []
        for r in range(batch.rows):
            q, k, v = workloads.new_tokens(wl, r, int(new[r]), int(past[r]))
            q_l.append(q); k_l.append(k); v_l.append(v)
            p_l.append(np.arange(past[r], past[r] + new[r], dtype=np.int32))
            s_l.append(np.full(int(new[r]), r, dtype=np.int32))
        self.h_q = torch.from_numpy(np.concatenate(q_l)).to(dt).pin_memory()
        self.h_k = torch.from_numpy(np.concatenate(k_l)).to(dt).pin_memory()
        self.h_v = torch.from_numpy(np.concatenate(v_l)).to(dt).pin_memory()
        self.h_pos = torch.from_numpy(np.concatenate(p_l)).pin_memory()
        self.h_sid = torch.from_numpy(np.concatenate(s_l)).pin_memory()
        self.h_table = torch.from_numpy(self.table_host).pin_memory()
        total = (past + new).astype(np.int32)
        self.h_lens = torch.from_numpy(total[nchunk:].copy()).pin_memory()
        cu = np.zeros(nchunk + 1, dtype=np.int32)
        cu[1:] = np.cumsum(new[:nchunk])
        self.h_cu = torch.from_numpy(cu).pin_memory()
        self.h_prefix = torch.from_numpy(past[:nchunk].astype(np.int32)).pin_memory()
        self.q = self.h_q.to(device)
        self.k = self.h_k.to(device)
        self.v = self.h_v.to(device)
        self.views = []
        if self.layers > 1:
            # each layer's fused QKV projection output [T, (Hq + 2 Hkv) D]: layer 0 holds this
            # step's tokens, the others fresh N(0,1) rows; q is rotated into the dense self.q
            T = self.h_q.shape[0]
            for l in range(self.layers):
                if l == 0:
                    x = torch.cat([self.q.reshape(T, -1), self.k.reshape(T, -1), self.v.reshape(T, -1)], 1)
                else:
                    x = torch.randn((T, (wl.num_q_heads + 2 * H) * D), generator=gen, device=device).to(dt)
                self.views.append(kv.split_qkv(x, wl.num_q_heads, H, D))
        self.pos = self.h_pos.to(device)
        self.sid = self.h_sid.to(device)
        self.lens = self.h_lens.to(device)
        self.cu = self.h_cu.to(device)
        self.prefix = self.h_prefix.to(device)
        self.n_dec = batch.rows - nchunk
        self.n_tok = int(new.sum())
        self.chunk_tokens = int(new[:nchunk].sum())
        self.max_len = int(total[nchunk:].max()) if self.n_dec else 1
        self.max_q = int(new[:nchunk].max()) if nchunk else 0
        self.q_dec = self.q[self.chunk_tokens:]
        self.q_pre = self.q[:self.chunk_tokens]
        self.out_dec = torch.empty_like(self.q_dec)
        self.out_pre = torch.empty_like(self.q_pre)
        self.d_table_dec = self.d_table[nchunk:]
        self.d_table_pre = self.d_table[:nchunk]
        self.splits = kv.decode_num_splits(self.cfg, self.n_dec, self.max_len, 0) if self.n_dec else 0
        nws = kv.decode_workspace_size(self.cfg, max(1, self.n_dec), self.max_len, 0)
        self.ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=device)
        # fp8 prefill: its bf16 copy of the chunks' blocks
        self.pre_kv_tokens = int(np.sum(total[:nchunk]))
        self.ws_pre = None
        if self.fp8 and nchunk:
            n = kv.prefill_fp8_workspace_size(self.cfg, BS, self.table_host.shape[1], nchunk, self.pre_kv_tokens)
            self.ws_pre = torch.empty(n, dtype=torch.uint8, device=device)
        self.h_out = torch.empty(self.out_dec.shape, dtype=dt).pin_memory()
        self.h_out_pre = torch.empty(self.out_pre.shape, dtype=dt).pin_memory()
        # algorithmic bytes / flops
        E = wl.elem_bytes
        Lr = self.layers
        self.kv_bytes_decode = Lr * workloads.kv_bytes_read(wl, total[nchunk:])
        if self.fp8:
            self.kv_bytes_decode = int(np.sum(total[nchunk:])) * 2 * H * (D + 4)
        self.kv_bytes_prefill = Lr * workloads.kv_bytes_read(wl, total[:nchunk])
        if self.fp8:
            self.kv_bytes_prefill = int(np.sum(total[:nchunk])) * 2 * H * (D + 4)
        self.rope_bytes = Lr * self.n_tok * 2 * (wl.num_q_heads + 2 * H) * D * E
        pre_flops = 0
        for c in range(nchunk):
            P, n = int(past[c]), int(new[c])
            pre_flops += 4 * D * wl.num_q_heads * int(np.sum(P + np.arange(n) + 1))
        self.prefill_flops = Lr * pre_flops
        self.launches_per_step = Lr * (1 + (1 if self.n_dec else 0) + (1 if self.splits > 1 else 0) +
                                       ((3 if self.fp8 else 1) if nchunk else 0))

    # host block allocator: hand out the blocks this step's tokens open, return them after
    def alloc_begin(self):
        if self.open_cells:
            ids = self.alloc.alloc(len(self.open_r))
            self.table_host[self.open_r, self.open_c] = ids
            return ids
        return None

    def alloc_end(self, ids):
        if ids is not None:
            self.alloc.free(ids[::-1])

    def _prefill(self, cache, q, cu, prefix, table, out):
        if self.fp8:
            self.kv.prefill_chunk_fp8(self.cfg, cache, q, cu, prefix, table, self.max_q, self.pre_kv_tokens, out=out,
                                      workspace=self.ws_pre)
        else:
            self.kv.prefill_chunk(self.cfg, cache, q, cu, prefix, table, self.max_q, out=out)

    def launch(self, ev=None):
        """One step: per layer rope_append, prefill_chunk, decode.  ev: per layer
        four events bracketing the three kernels."""
        kv = self.kv
        ids = self.alloc_begin()
        for l, cache in enumerate(self.caches):
            e = ev[l] if ev is not None else None
            if e is not None:
                e[0].record()
            if self.fp8:
                kv.rope_append_fp8(self.cfg, cache, self.q, self.k, self.v, self.pos, self.sid, self.d_table)
            elif self.views:
                q, k, v = self.views[l]
                kv.rope_append(self.cfg, cache, q, k, v, self.pos, self.sid, self.d_table, q_out=self.q)
            else:
                kv.rope_append(self.cfg, cache, self.q, self.k, self.v, self.pos, self.sid, self.d_table)
            if e is not None:
                e[1].record()
            if self.nchunk:
                self._prefill(cache, self.q_pre, self.cu, self.prefix, self.d_table_pre, self.out_pre)
            if e is not None:
                e[2].record()
            if self.n_dec:
                (kv.decode_fp8 if self.fp8 else kv.decode)(self.cfg, cache, self.q_dec, self.d_table_dec, self.lens,
                                                            self.max_len, out=self.out_dec, workspace=self.ws)
            if e is not None:
                e[3].record()
        self.alloc_end(ids)

    def _host_inputs(self, b=0):
        return {"q": self.h_q, "k": self.h_k, "v": self.h_v, "pos": self.h_pos, "sid": self.h_sid,
                "table": self.h_tables[b], "lens": self.h_lens, "cu": self.h_cu, "prefix": self.h_prefix}

    def e2e_setup(self):
        """Two device buffer sets and a copy stream: step i+1's inputs go up and
        step i-1's outputs come down while step i computes."""
        torch = self.torch
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        self.h_tables = [torch.from_numpy(self.table_host.copy()).pin_memory() for _ in range(2)]
        self.bufs = []
        for b in range(2):
            d = {n: torch.empty(h.shape, dtype=h.dtype, device=self.dev) for n, h in self._host_inputs(b).items()}
            d["out_dec"] = torch.empty_like(self.out_dec)
            d["out_pre"] = torch.empty_like(self.out_pre)
            d["q_dec"] = d["q"][self.chunk_tokens:]
            d["q_pre"] = d["q"][:self.chunk_tokens]
            d["table_dec"] = d["table"][self.nchunk:]
            d["table_pre"] = d["table"][:self.nchunk]
            self.bufs.append(d)
        self.h_outs = [(torch.empty(self.out_dec.shape, dtype=self.dt).pin_memory(),
                        torch.empty(self.out_pre.shape, dtype=self.dt).pin_memory()) for _ in range(2)]
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]

    def _upload(self, i):
        torch, xs, b = self.torch, self.copy_stream, i % 2
        ids = self.alloc_begin()                       # host allocator work of step i
        self.h_tables[b].copy_(torch.from_numpy(self.table_host))
        self.alloc_end(ids)
        with torch.cuda.stream(xs):
            if i >= 2:
                xs.wait_event(self.ev_done[b])         # step i-2 no longer reads buffer b
            for n, h in self._host_inputs(b).items():
                self.bufs[b][n].copy_(h, non_blocking=True)
            self.ev_in[b].record(xs)

    def run_e2e(self, steps: int) -> float:
        """`steps` steps end to end through the C ABI from pinned host buffers;
        returns seconds from the first upload to the last download."""
        torch, kv, xs = self.torch, self.kv, self.copy_stream
        cs = torch.cuda.current_stream()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(xs)
        self._upload(0)
        for i in range(steps):
            b = i % 2
            d = self.bufs[b]
            if i + 1 < steps:
                self._upload(i + 1)
            cs.wait_event(self.ev_in[b])
            (kv.rope_append_fp8 if self.fp8 else kv.rope_append)(self.cfg, self.cache, d["q"], d["k"], d["v"],
                                                                  d["pos"], d["sid"], d["table"])
            if self.nchunk:
                self._prefill(self.cache, d["q_pre"], d["cu"], d["prefix"], d["table_pre"], d["out_pre"])
            if self.n_dec:
                (kv.decode_fp8 if self.fp8 else kv.decode)(self.cfg, self.cache, d["q_dec"], d["table_dec"],
                                                            d["lens"], self.max_len, out=d["out_dec"],
                                                            workspace=self.ws)
            self.ev_done[b].record(cs)
            with torch.cuda.stream(xs):
                xs.wait_event(self.ev_done[b])
                if self.n_dec:
                    self.h_outs[b][0].copy_(d["out_dec"], non_blocking=True)
                if self.nchunk:
                    self.h_outs[b][1].copy_(d["out_pre"], non_blocking=True)
        end.record(xs)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    def h2d_bytes(self) -> int:
        return int(sum(t.numel() * t.element_size() for t in self._host_inputs(0).values()))

    def d2h_bytes(self) -> int:
        n = int(self.h_out.numel() * self.h_out.element_size()) if self.n_dec else 0
        return n + (int(self.h_out_pre.numel() * self.h_out_pre.element_size()) if self.nchunk else 0)


def oracle_sample(wl: workloads.Workload, target_s: float = 12.0, max_rows: int = 8):
    """Times the oracle (as it stands) on a bounded sample of the workload's decode rows:
    RoPE + rounding + append of each row's new token, then attention of its query.
    Returns (GB/s of KV bytes, cores, sample description, per-pass seconds)."""
    import oracle

    batch = workloads.make_batch(wl, num_blocks=1 << 22)
    dec = list(range(wl.chunks, batch.rows))
    rows = dec[:max_rows]
    BS, H, D = wl.block_size, wl.num_kv_heads, wl.head_dim
    need = [(int(batch.total[r]) + BS - 1) // BS for r in rows]
    table = np.full((len(rows), max(need)), -1, dtype=np.int32)
    o = 0
    for i, n in enumerate(need):
        table[i, :n] = np.arange(o, o + n, dtype=np.int32)
        o += n
    cache = oracle.Cache(o, BS, H, D)
    od = oracle.BF16 if wl.dtype == "bf16" else oracle.F32
    for i, r in enumerate(rows):
        p = int(batch.past[r])
        k, v = workloads.history(wl, r, p)
        oracle.append(cache, oracle.round_to(k, od), oracle.round_to(v, od), np.arange(p), np.full(p, i, np.int32),
                      table)
    news = [workloads.new_tokens(wl, r, 1, int(batch.past[r])) for r in rows]
    kvb = workloads.kv_bytes_read(wl, batch.total[rows])

    def one_pass():
        qs = []
        for i, r in enumerate(rows):
            p = int(batch.past[r])
            q, k, v = news[i]
            kh = oracle.round_to(oracle.rope(k.astype(np.float64), [p]), od)
            oracle.append(cache, kh, oracle.round_to(v, od), [p], [i], table)
            qs.append(oracle.round_to(oracle.rope(q.astype(np.float64), [p]), od)[0])
        oracle.attend(cache, np.stack(qs), list(range(len(rows))), [int(batch.past[r]) for r in rows], table,
                      wl.num_q_heads)

    t0 = time.perf_counter()
    one_pass()
    t1 = time.perf_counter()
    return kvb, oracle.num_cores(), f"{len(rows)} decode rows of {wl.key} (their lengths, all heads)", t1 - t0, one_pass


def cpu_baseline(wl, target_s: float = 12.0):
    kvb, cores, desc, t_one, one_pass = oracle_sample(wl)
    reps = max(1, min(200, int(target_s / max(t_one, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(reps):
        one_pass()
    dt = time.perf_counter() - t0
    return {"value": kvb * reps / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{desc}, {reps} passes in {dt:.1f} s (fp64 C, {cores} threads)"}


def graph_timings(st, dev, reps: int = 50, replays: int = 5, flushed_steps: int = 20):
    """Launch-bound workloads: the step as CUDA-graph replays of `reps` steps
    (median over `replays`, L2 warm), and single eager steps each after writing
    a buffer twice the L2 size (median, L2 cold).  The host allocator work of a
    step is not replayed by the graph (no blocks change hands in these
    contiguous-cache workloads)."""
    import torch

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            st.launch()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            st.launch()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(replays):
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / reps)
    flush = torch.empty(2 * 129 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    cold = []
    for _ in range(flushed_steps):
        flush.fill_(1.0)
        a.record()
        st.launch()
        b.record()
        torch.cuda.synchronize()
        cold.append(a.elapsed_time(b))
    status = st.kv.get_device_status()
    if status:
        raise RuntimeError(f"device status {st.kv.STATUS.get(status)} in the graph timings")
    return {"ms_per_step_l2_warm": statistics.median(times), "reps_per_replay": reps, "replays": replays,
            "ms_per_step_l2_flushed": statistics.median(cold), "flushed_steps": flushed_steps,
            "launches_per_step": st.launches_per_step}


def time_steps(st, steps: int, warmup: int, dev):
    """Eager steps of `st` with per-kernel CUDA events on the launching stream and
    the clocks sampled meanwhile: (seconds, per-step ms of rope_append, prefill,
    decode summed over layers, clocks)."""
    import torch

    for _ in range(max(3, warmup)):
        st.launch()
    torch.cuda.synchronize()
    status = st.kv.get_device_status()
    if status:
        raise RuntimeError(f"device status {st.kv.STATUS.get(status)} after warm-up")
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(st.layers)]
           for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev)
    torch.cuda.synchronize()
    clocks.start()
    start.record()
    for i in range(steps):
        st.launch(evs[i])
    end.record()
    torch.cuda.synchronize()
    ck = clocks.stop()
    status = st.kv.get_device_status()
    if status:
        raise RuntimeError(f"device status {st.kv.STATUS.get(status)} in the timed region")
    ms = [statistics.mean(sum(e[a].elapsed_time(e[a + 1]) for e in es) for es in evs) for a in range(3)]
    return start.elapsed_time(end) / 1e3, ms, ck


def per_config(dev, steps: int, warmup: int, hbm: float, bf16_burst: float, peak_src: str):
    """The other workloads, measured in the same run as the headline step, one
    at a time (each freed before the next): the decode-only configs (decode
    split + combine time, KV GB/s and fraction of the measured HBM peak; c4 on
    its 180e9-byte pool, halved until it fits, the size used recorded), c4 over
    an fp8 cache, c4 with groups of 8 and of 2 query heads (the same KV bytes), the
    launch-bound GPT-2-shape configs as CUDA-graph replays, the mixed step
    over an fp8 cache, and the mixed step over 32 layers."""
    import torch

    res = {}
    plan = [("c3", {}), ("c4", {}), ("c4g8", {}), ("c4g2", {}), ("c4_fp8", {"kv_fp8": True}), ("c5_fp8", {"kv_fp8": True}),
            ("c1_graph", {}), ("c2_graph", {}), ("c5_32layers", {"layers": 32})]
    for name, kw in plan:
        key = name.split("_")[0]
        wl = workloads.WORKLOADS[key]
        try:
            st = Step(wl, dev, **kw)
        except torch.OutOfMemoryError as e:
            res[name] = {"skipped": f"out of device memory: {str(e).splitlines()[0]}"}
            torch.cuda.empty_cache()
            continue
        rec = {"workload": f"{wl.key}: {wl.name}", "pool_bytes": st.pool_bytes, "layers": st.layers,
               "decode_splits": st.splits, "launches_per_step": st.launches_per_step}
        if name.endswith("_graph"):
            rec.update(graph_timings(st, dev))
            rec["kv_bytes_per_step"] = st.kv_bytes_decode
        else:
            n = max(5, min(steps, 100 if st.layers == 1 else 10))   # bounded: a 32-layer step takes ~26 ms
            secs, (t_rope, t_pre, t_dec), ck = time_steps(st, n, warmup, dev)
            rec.update({"steps": n, "ms_per_step": 1e3 * secs / n,
                        "kernels_ms": {"rope_append": t_rope, "prefill": t_pre, "decode": t_dec},
                        "clocks": ck})
            if st.fp8:
                rec["kv_cache"] = "e4m3 codes + one fp32 scale per (slot, KV head); kv bytes count both"
            if st.n_dec:
                gbs = st.kv_bytes_decode / (t_dec / 1e3) / 1e9
                rec.update({"decode_kv_bytes": st.kv_bytes_decode, "decode_kv_gbs": gbs,
                            "decode_hbm_frac": gbs / hbm, "peak_source": f"hbm_gbs, {peak_src}"})
            if st.nchunk:
                tf = st.prefill_flops / (t_pre / 1e3) / 1e12
                rec.update({"prefill_tflops": tf, "prefill_frac": tf / bf16_burst,
                            "prefill_peak_source": f"bf16_tflops (burst), {peak_src}"})
            rec["value_gbs"] = (st.kv_bytes_decode + st.kv_bytes_prefill) * n / secs / 1e9
        res[name] = rec
        del st
        torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world):
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = workloads.WORKLOADS[args.workload]
    st = Step(wl, dev, rows=args.rows, compact_pool=args.compact_pool, chunks=args.chunks, layers=args.layers,
              kv_fp8=args.kv_dtype == "fp8")
    hbm, bf16_burst, bf16_sus, peak_src = peaks()
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        st.launch()
    torch.cuda.synchronize()
    status = st.kv.get_device_status()
    if status:
        raise RuntimeError(f"device status {st.kv.STATUS.get(status)} after warm-up")
    K = args.steps
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(st.layers)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    start.record(stream)
    for i in range(K):
        st.launch(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    ck = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    elapsed = start.elapsed_time(end) / 1e3
    # per step: summed over the step's layers
    t_rope = statistics.mean(sum(e[0].elapsed_time(e[1]) for e in es) for es in evs) / 1e3
    t_pre = statistics.mean(sum(e[1].elapsed_time(e[2]) for e in es) for es in evs) / 1e3
    t_dec = statistics.mean(sum(e[2].elapsed_time(e[3]) for e in es) for es in evs) / 1e3
    status = st.kv.get_device_status()
    if status:
        raise RuntimeError(f"device status {st.kv.STATUS.get(status)} in the timed region")
    graph = graph_timings(st, dev) if args.graph else None
    # e2e through host buffers
    e2e = None
    e2e_t = 0.0
    if not args.no_e2e and st.layers == 1:
        st.e2e_setup()
        st.run_e2e(3)  # warm-up
        e2e_t = st.run_e2e(K)
    elapsed, e2e_t = max_over_ranks([elapsed, e2e_t], dev)
    step_bytes = st.kv_bytes_decode + st.kv_bytes_prefill
    value = whole_job_rate(step_bytes, K, world, elapsed) / 1e9
    if not args.no_e2e and st.layers == 1:
        e2e = {"value": whole_job_rate(step_bytes, K, world, e2e_t) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": st.h2d_bytes(),
               "d2h_bytes_per_step": st.d2h_bytes(), "ms_per_step": 1e3 * e2e_t / K}
    # dominant kernel roofline (and the decode kernel's, the HBM-bound part)
    parts = {"decode": t_dec, "prefill": t_pre, "rope_append": t_rope}
    dom = max(parts, key=parts.get)

    # the tensor peak that applies: a kernel timed inside a region shorter than
    # a second runs before the power cap settles (burst figure), a longer one
    # after (sustained figure)
    if elapsed < 1.0:
        bf16_peak, bf16_src = bf16_burst, f"bf16_tflops (burst: timed region {elapsed:.3f} s < 1 s), {peak_src}"
    else:
        bf16_peak, bf16_src = bf16_sus, f"bf16_tflops_sustained (timed region {elapsed:.2f} s >= 1 s), {peak_src}"

    def roof_of(k):
        if k == "prefill":
            ach = st.prefill_flops / t_pre / 1e12
            kname = "prefill_fp8_plan+prefill_fp8_expand+prefill_chunk" if st.fp8 else "prefill_chunk"
            return {"kernel": kname, "bound": "tensor", "achieved": ach, "peak": bf16_peak,
                    "unit": "TFLOP/s", "frac": ach / bf16_peak,
                    "traffic": None if st.fp8 else measured_traffic("prefill_chunk", wl.key),
                    "peak_source": bf16_src}
        name = "decode_split+decode_combine" if k == "decode" else "rope_append"
        by = st.kv_bytes_decode if k == "decode" else st.rope_bytes
        ach = by / parts[k] / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": measured_traffic(name, wl.key + ("-fp8" if st.fp8 else "")),
                "peak_source": f"hbm_gbs, {peak_src}"}

    roof = roof_of(dom)
    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": 1e3 * elapsed / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 q/out, e4m3 KV" if st.fp8 else wl.dtype, "data": "synthetic",
        "config": {"workload": f"{wl.key}: {wl.name}" + (f" (first {args.rows} decode rows)" if args.rows else ""),
                   "decode_seqs": st.n_dec, "prefill_chunks": st.nchunk,
                   "query_tokens": st.n_tok, "q_heads": wl.num_q_heads, "kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "block_size": wl.block_size, "pool_bytes": st.pool_bytes,
                   "kv_bytes_per_step": step_bytes, "decode_splits": st.splits,
                   "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB of KV per step)"
                   if step_bytes > 2e8 else "L2-resident: KV smaller than L2, not flushed",
                   "parallelism": f"replicas x{world}",
                   "layers": st.layers,
                   **({"kv_cache": "e4m3 codes + one fp32 scale per (slot, KV head); kv_bytes count both"}
                      if st.fp8 else {}),
                   **({"qkv_input": "per layer: views of its fused [T, (Hq+2Hkv)D] QKV output; q rotated into "
                                    "a dense buffer; no host upload (e2e measured at layers=1)"}
                      if st.layers > 1 else {})},
        "query_tokens_per_s": whole_job_rate(st.n_tok, K, world, elapsed),
        "hbm_frac": (st.kv_bytes_decode / t_dec / 1e9) / hbm if st.n_dec else None,
        "kernels_ms": {k: 1e3 * v for k, v in parts.items()},
        "decode_kv_gbs": st.kv_bytes_decode / t_dec / 1e9 if st.n_dec else None,
        "roofline": roof,
        "roofline_decode": roof_of("decode") if st.n_dec and dom != "decode" else None,
        "roofline_rope_append": roof_of("rope_append") if dom != "rope_append" else None,
        "e2e": e2e,
        "gpu_launches": K * st.launches_per_step,
        "clocks": ck,
        **({"graph": graph} if graph else {}),
    }
    if st.nchunk:
        out["prefill_tflops"] = st.prefill_flops / t_pre / 1e12
    if not args.no_per_config and args.workload == DEFAULT_WORKLOAD and not (args.rows or args.chunks >= 0 or
                                                                             args.compact_pool or st.fp8 or
                                                                             st.layers > 1):
        del st
        torch.cuda.empty_cache()
        out["per_config"] = per_config(dev, K, args.warmup, hbm, bf16_burst, peak_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl)
    return out


def run_reference(args, world):
    """The fp64 oracle as it stands, on this host's cores, same metric and workload."""
    wl = workloads.WORKLOADS[args.workload]
    kvb, cores, desc, _, one_pass = oracle_sample(wl)
    for _ in range(args.warmup):
        one_pass()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_pass()
    dt = time.perf_counter() - t0
    v = kvb * args.steps / dt / 1e9
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl.key}: {wl.name}", "sample": desc},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return
    if world > 1:
        import torch

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group(backend="nccl")
    out = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
