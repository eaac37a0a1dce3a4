"""Shared set-up of GPU parity cases: builds the same KV cache on the GPU (the
library's documented layout) and in the fp64 oracle (its own slot-major
layout) from the seeded inputs of workloads.py, runs the library through its
C ABI, and compares with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import kv_cache_attention_rope_gb300 as kv
import oracle
import workloads

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
KV_DT = {"bf16": kv.BF16, "f32": kv.F32}
OR_DT = {"bf16": oracle.BF16, "f32": oracle.F32}
# attention tolerances: max abs and relative L2
TOL = {"bf16": (1e-2, 5e-3), "f32": (1e-5, 1e-5)}


def f64(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def put_rows(pool: torch.Tensor, table_row: np.ndarray, positions: np.ndarray, rows: torch.Tensor) -> None:
    """Writes rows[n] (Hkv x D) at token positions[n] of the sequence owning table_row.

    The library's documented layout: pool[block][kv_head][offset][d] with
    block = table_row[p // block_size], offset = p % block_size.
    """
    BS = pool.shape[2]
    blk = torch.from_numpy(table_row[positions // BS].astype(np.int64)).to(pool.device)
    off = torch.from_numpy((positions % BS).astype(np.int64)).to(pool.device)
    pool[blk, :, off, :] = rows.to(pool.dtype)


def get_rows(pool: torch.Tensor, table_row: np.ndarray, positions: np.ndarray) -> torch.Tensor:
    BS = pool.shape[2]
    blk = torch.from_numpy(table_row[positions // BS].astype(np.int64)).to(pool.device)
    off = torch.from_numpy((positions % BS).astype(np.int64)).to(pool.device)
    return pool[blk, :, off, :]


def compare(got: np.ndarray, ref: np.ndarray, dtype: str, what: str):
    atol, rtol = TOL[dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref).max() if got.size else 0.0
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got - ref)
    assert err <= atol and rel <= rtol, f"{what}: max abs {err:.3e} (<= {atol}), rel L2 {rel:.3e} (<= {rtol})"
    return err, rel


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (at least the smallest normal's spacing)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    e = np.floor(np.log2(ax))
    return 2.0 ** (e - 7)


def ulp_f32(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    e = np.floor(np.log2(ax))
    return 2.0 ** (e - 23)


def check_rotation(got: np.ndarray, exact: np.ndarray, dtype: str, what: str) -> int:
    """Every element within 1 ulp of the exact rotation; returns how many differ
    from the correctly rounded value (expected: none)."""
    ulp = ulp_bf16(exact) if dtype == "bf16" else ulp_f32(exact)
    bad = np.abs(got - exact) > ulp
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1 ulp, worst {np.abs(got - exact)[bad].max():.3e}"
    rn = oracle.round_to(exact, OR_DT[dtype])
    return int((got != rn).sum())


class DecodeCase:
    """One decode step of a workload: cache history, new token, expected output.

    rows_checked: rows whose history comes from workloads.history (CPU, seeded)
    and that the oracle recomputes; every other row's history is drawn on the
    device with torch.randn (it only has to exist and be finite).
    """

    def __init__(self, wl: workloads.Workload, batch: workloads.Batch, rows_checked, device="cuda",
                 fill_nan=True):
        self.wl, self.batch, self.device = wl, batch, torch.device(device)
        self.rows = sorted(int(r) for r in rows_checked)
        dt = TORCH_DT[wl.dtype]
        nb, BS, H, D = batch.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim
        self.cache = kv.Cache.empty(nb, H, BS, D, dt, self.device)
        if fill_nan:
            self.cache.k_pool.fill_(float("nan"))
            self.cache.v_pool.fill_(float("nan"))
        self.cfg = kv.make_config(wl.num_q_heads, H, D, KV_DT[wl.dtype])
        # oracle cache over the checked rows only, blocks renumbered compactly
        need = [(int(batch.total[r]) + BS - 1) // BS for r in self.rows]
        self.o_table = np.full((len(self.rows), max(need) if need else 1), -1, dtype=np.int32)
        nxt = 0
        for i, n in enumerate(need):
            self.o_table[i, :n] = np.arange(nxt, nxt + n, dtype=np.int32)
            nxt += n
        self.ocache = oracle.Cache(max(nxt, 1), BS, H, D)
        gen = torch.Generator(device=self.device)
        gen.manual_seed(1234)
        for r in range(batch.rows):
            past = int(batch.past[r])
            if past == 0:
                continue
            pos = np.arange(past)
            if r in self.rows:
                k, v = workloads.history(wl, r, past)
                kt, vt = torch.from_numpy(k).to(dt), torch.from_numpy(v).to(dt)
                put_rows(self.cache.k_pool, batch.block_table[r], pos, kt.to(self.device))
                put_rows(self.cache.v_pool, batch.block_table[r], pos, vt.to(self.device))
                i = self.rows.index(r)
                oracle.append(self.ocache, kt.double().numpy(), vt.double().numpy(), pos,
                              np.full(past, i, np.int32), self.o_table)
            else:
                kt = torch.randn((past, H, D), generator=gen, device=self.device, dtype=torch.float32)
                vt = torch.randn((past, H, D), generator=gen, device=self.device, dtype=torch.float32)
                put_rows(self.cache.k_pool, batch.block_table[r], pos, kt)
                put_rows(self.cache.v_pool, batch.block_table[r], pos, vt)
        # new tokens, one per row
        qs, ks, vs = [], [], []
        for r in range(batch.rows):
            q, k, v = workloads.new_tokens(wl, r, 1, int(batch.past[r]))
            qs.append(q[0]); ks.append(k[0]); vs.append(v[0])
        self.q_raw = torch.from_numpy(np.stack(qs)).to(dt)
        self.k_raw = torch.from_numpy(np.stack(ks)).to(dt)
        self.v_raw = torch.from_numpy(np.stack(vs)).to(dt)
        self.d_table = torch.from_numpy(batch.block_table).to(self.device)
        self.positions = torch.from_numpy(batch.past.astype(np.int32)).to(self.device)
        self.seq_ids = torch.arange(batch.rows, dtype=torch.int32, device=self.device)
        self.seq_lens = torch.from_numpy(batch.total.astype(np.int32)).to(self.device)
        self.max_len = int(batch.total.max())

    def run(self, num_splits=0, q=None):
        """rope_append of the new tokens, then decode; returns (q_rotated, out) on the device."""
        q = self.q_raw.to(self.device).clone() if q is None else q
        kv.rope_append(self.cfg, self.cache, q, self.k_raw.to(self.device), self.v_raw.to(self.device),
                       self.positions, self.seq_ids, self.d_table)
        out = kv.decode(self.cfg, self.cache, q, self.d_table, self.seq_lens, self.max_len,
                        num_splits=num_splits)
        return q, out

    def expected(self):
        """Oracle: rotated+rounded new k appended, attention of the rotated+rounded q."""
        od = OR_DT[self.wl.dtype]
        qh, outs = [], None
        for i, r in enumerate(self.rows):
            p = int(self.batch.past[r])
            kh = oracle.round_to(oracle.rope(self.k_raw[r:r + 1].double().numpy(), [p]), od)
            oracle.append(self.ocache, kh, self.v_raw[r:r + 1].double().numpy(), [p], [i], self.o_table)
            qh.append(oracle.round_to(oracle.rope(self.q_raw[r:r + 1].double().numpy(), [p]), od)[0])
        pos = [int(self.batch.past[r]) for r in self.rows]
        outs = oracle.attend(self.ocache, np.stack(qh), list(range(len(self.rows))), pos, self.o_table,
                             self.wl.num_q_heads)
        return np.stack(qh), outs


class PrefillCase:
    """Chunks of new query tokens over cached prefixes: the chunk tokens go
    through rope_append (GPU) and rope + round + append (oracle); history
    tokens before each prefix are drawn N(0,1) and written to both caches."""

    def __init__(self, hq, hkv, prefixes, qlens, block_size=16, seed=0, device="cuda", k_scale=None,
                 extra_blocks=5, head_dim=128):
        D = head_dim
        self.hq, self.hkv, self.D = hq, hkv, D
        self.prefixes = np.asarray(prefixes, dtype=np.int64)
        self.qlens = np.asarray(qlens, dtype=np.int64)
        n = len(prefixes)
        BS = block_size
        total = self.prefixes + self.qlens
        need = (total + BS - 1) // BS
        nb = int(need.sum()) + extra_blocks
        g = np.random.default_rng(seed)
        perm = g.permutation(nb).astype(np.int32)
        table = np.full((n, int(need.max())), -1, dtype=np.int32)
        o = 0
        for r, k in enumerate(need):
            table[r, :k] = perm[o:o + k]
            o += k
        self.table = table
        self.device = torch.device(device)
        self.cfg = kv.make_config(hq, hkv, D, kv.BF16)
        self.cache = kv.Cache.empty(nb, hkv, BS, D, torch.bfloat16, self.device)
        self.cache.k_pool.fill_(float("nan"))
        self.cache.v_pool.fill_(float("nan"))
        self.ocache = oracle.Cache(nb, BS, hkv, D)
        for r in range(n):
            P = int(self.prefixes[r])
            if P:
                k = torch.from_numpy(g.standard_normal((P, hkv, D), dtype=np.float32)).to(torch.bfloat16)
                v = torch.from_numpy(g.standard_normal((P, hkv, D), dtype=np.float32)).to(torch.bfloat16)
                put_rows(self.cache.k_pool, table[r], np.arange(P), k.to(self.device))
                put_rows(self.cache.v_pool, table[r], np.arange(P), v.to(self.device))
                oracle.append(self.ocache, k.double().numpy(), v.double().numpy(), np.arange(P),
                              np.full(P, r, np.int32), table)
        T = int(self.qlens.sum())
        self.q_raw = torch.from_numpy(g.standard_normal((T, hq, D), dtype=np.float32)).to(torch.bfloat16)
        k_raw = g.standard_normal((T, hkv, D), dtype=np.float32)
        if k_scale is not None:
            k_raw = k_raw * k_scale(np.arange(T))[:, None, None]
        self.k_raw = torch.from_numpy(k_raw).to(torch.bfloat16)
        self.v_raw = torch.from_numpy(g.standard_normal((T, hkv, D), dtype=np.float32)).to(torch.bfloat16)
        self.pos = np.concatenate([np.arange(p, p + q) for p, q in zip(self.prefixes, self.qlens)]).astype(np.int32)
        self.seq = np.concatenate([np.full(q, r) for r, q in enumerate(self.qlens)]).astype(np.int32)
        self.cu = np.zeros(n + 1, dtype=np.int32)
        self.cu[1:] = np.cumsum(self.qlens)

    def run(self):
        dev = self.device
        q = self.q_raw.to(dev).contiguous()
        d_table = torch.from_numpy(self.table).to(dev)
        kv.rope_append(self.cfg, self.cache, q, self.k_raw.to(dev), self.v_raw.to(dev),
                       torch.from_numpy(self.pos).to(dev), torch.from_numpy(self.seq).to(dev), d_table)
        out = kv.prefill_chunk(self.cfg, self.cache, q, torch.from_numpy(self.cu).to(dev),
                               torch.from_numpy(self.prefixes.astype(np.int32)).to(dev), d_table,
                               int(self.qlens.max()))
        return q, out

    def expected(self, rows=None):
        """Oracle output for the given query rows (indices into the chunk tokens)."""
        od = oracle.BF16
        kh = oracle.round_to(oracle.rope(self.k_raw.double().numpy(), self.pos), od)
        oracle.append(self.ocache, kh, self.v_raw.double().numpy(), self.pos, self.seq, self.table)
        rows = np.arange(len(self.pos)) if rows is None else np.asarray(rows)
        qh = oracle.round_to(oracle.rope(self.q_raw[rows].double().numpy(), self.pos[rows]), od)
        return rows, oracle.attend(self.ocache, qh, self.seq[rows], self.pos[rows], self.table, self.hq)
