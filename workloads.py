"""Seeded synthetic inputs for the RoPE + KV-cache + attention path.

This module is shared by the tests (which feed the same arrays to the CUDA
library and to the fp64 oracle) and by bench.py.  It holds no arithmetic of
the method: it only draws numbers (N(0,1) vectors, integer lengths, block
permutations) and states the workload shapes.  The shapes follow the models
the pages use as examples: GPT-2 (12 heads x 64), a Qwen/Llama-style model
(32 heads x 128, hidden 4096) and its grouped-query variant (32 query heads /
8 KV heads).  No public dataset is involved.

Seeds: q/k/v data 0, lengths 1, block permutation 2.  Every array is a numpy
array; callers move it to a device themselves.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

DATA_SEED = 0
LEN_SEED = 1
PERM_SEED = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    name: str
    dtype: str              # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    layout: str             # "contiguous" or "paged"
    block_size: int         # 16 for paged; max_len for contiguous
    decode_batch: int       # decode sequences
    decode_len: tuple       # inclusive range of PAST lengths; the new token sits at position len
    chunks: int = 0         # prefill chunks
    chunk_len: int = 0      # query tokens per chunk
    prefix_len: tuple = (0, 0)
    pool_bytes: int = 0     # K+V bytes of the paged pool (0: twice what the sequences need)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    "c1": Workload("c1", "tiny decode fp32, GPT-2 shape 12x64, contiguous, 127 past tokens",
                   "f32", 12, 12, 64, "contiguous", 128, 1, (127, 127)),
    "c2": Workload("c2", "GPT-2 shape decode bf16, batch 8, 12x64, contiguous, past len U[1,1024]",
                   "bf16", 12, 12, 64, "contiguous", 1025, 8, (1, 1024)),
    "c3": Workload("c3", "Qwen-shape MHA decode bf16, batch 64, 32x128, paged 16, past len U[512,4096]",
                   "bf16", 32, 32, 128, "paged", 16, 64, (512, 4096)),
    "c4": Workload("c4", "GQA decode bf16, batch 256, 32q/8kv x128, paged 16 over a 180e9-byte pool, "
                   "past len U[1024,8192]",
                   "bf16", 32, 8, 128, "paged", 16, 256, (1024, 8192), pool_bytes=180 * 10**9),
    # c4 with groups of 8 query heads per KV head: the same KV bytes as c4, twice the queries
    "c4g8": Workload("c4g8", "GQA-8 decode bf16, batch 256, 64q/8kv x128, paged 16 over a 180e9-byte pool, "
                     "past len U[1024,8192]",
                     "bf16", 64, 8, 128, "paged", 16, 256, (1024, 8192), pool_bytes=180 * 10**9),
    # c4 with groups of 2 query heads per KV head (the CUDA-core decode path): the same KV bytes as c4
    "c4g2": Workload("c4g2", "GQA-2 decode bf16, batch 256, 16q/8kv x128, paged 16 over a 180e9-byte pool, "
                     "past len U[1024,8192]",
                     "bf16", 16, 8, 128, "paged", 16, 256, (1024, 8192), pool_bytes=180 * 10**9),
    "c5": Workload("c5", "mixed: 16 prefill chunks x 512 causal queries over prefix U[0,8192] + 128 decode "
                   "seqs past len U[256,8192], GQA 32q/8kv x128, paged 16",
                   "bf16", 32, 8, 128, "paged", 16, 128, (256, 8192),
                   chunks=16, chunk_len=512, prefix_len=(0, 8192)),
}


def rng(*stream: int) -> np.random.Generator:
    return np.random.default_rng(list(stream))


def normal(shape, *stream: int) -> np.ndarray:
    """Standard-normal float32 array from the counter-free PCG64 stream `stream`."""
    return rng(*stream).standard_normal(size=shape, dtype=np.float32)


@dataclasses.dataclass
class Batch:
    """Sequences of one step.  Row r of the block table belongs to sequence r.

    past[r]   tokens already in the cache (positions 0..past[r]-1)
    new[r]    tokens appended this step (positions past[r]..past[r]+new[r]-1)
    kind[r]   "decode" (new == 1) or "prefill" (a chunk of new >= 1 queries)
    """
    wl: Workload
    past: np.ndarray
    new: np.ndarray
    kind: list
    num_blocks: int
    block_table: np.ndarray     # [rows, max_blocks] int32, -1 where unused

    @property
    def rows(self) -> int:
        return len(self.past)

    @property
    def total(self) -> np.ndarray:
        return self.past + self.new


def lengths(wl: Workload) -> tuple[np.ndarray, np.ndarray]:
    """(decode past lengths [decode_batch], prefill prefixes [chunks]), inclusive uniform integers."""
    g = rng(LEN_SEED)
    dec = g.integers(wl.decode_len[0], wl.decode_len[1] + 1, size=wl.decode_batch).astype(np.int64)
    pre = np.zeros(0, dtype=np.int64)
    if wl.chunks:
        pre = rng(LEN_SEED, 1).integers(wl.prefix_len[0], wl.prefix_len[1] + 1,
                                         size=wl.chunks).astype(np.int64)
    return dec, pre


def make_batch(wl: Workload, num_blocks: int | None = None, rows_subset=None) -> Batch:
    """Lengths and block table of the workload (prefill chunks first, then decode rows)."""
    dec, pre = lengths(wl)
    past = np.concatenate([pre, dec])
    new = np.concatenate([np.full(len(pre), wl.chunk_len, dtype=np.int64),
                          np.ones(len(dec), dtype=np.int64)])
    kind = ["prefill"] * len(pre) + ["decode"] * len(dec)
    if rows_subset is not None:
        idx = np.asarray(rows_subset)
        past, new, kind = past[idx], new[idx], [kind[i] for i in idx]
    total = past + new
    BS = wl.block_size
    if wl.layout == "contiguous":
        if total.max() > BS:
            raise ValueError("contiguous row shorter than a sequence")
        nb = len(total) if num_blocks is None else int(num_blocks)
        perm = rng(PERM_SEED).permutation(nb)[: len(total)]
        table = perm.astype(np.int32).reshape(-1, 1)
        return Batch(wl, past, new, kind, nb, table)
    need = (total + BS - 1) // BS
    if num_blocks is None:
        if wl.pool_bytes:
            per_block = 2 * BS * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
            num_blocks = wl.pool_bytes // per_block
        else:
            num_blocks = int(2 * need.sum())
    if need.sum() > num_blocks:
        raise ValueError("pool too small for the batch")
    perm = rng(PERM_SEED).permutation(int(num_blocks))[: int(need.sum())].astype(np.int32)
    maxb = int(need.max())
    table = np.full((len(total), maxb), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[off:off + n]
        off += n
    return Batch(wl, past, new, kind, int(num_blocks), table)


def new_tokens(wl: Workload, row: int, n: int, past: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Raw q[n,Hq,D], k[n,Hkv,D], v[n,Hkv,D] (float32, N(0,1)) of `row`'s new tokens."""
    g = rng(DATA_SEED, 1, row)
    q = g.standard_normal((n, wl.num_q_heads, wl.head_dim), dtype=np.float32)
    k = g.standard_normal((n, wl.num_kv_heads, wl.head_dim), dtype=np.float32)
    v = g.standard_normal((n, wl.num_kv_heads, wl.head_dim), dtype=np.float32)
    return q, k, v


def history(wl: Workload, row: int, past: int) -> tuple[np.ndarray, np.ndarray]:
    """Cached K and V of positions 0..past-1 of `row`, as float32 N(0,1) [past, Hkv, D].

    Rotating i.i.d. N(0,1) pairs gives i.i.d. N(0,1) pairs again, so drawing the
    cached (already rotated) keys directly has the exact distribution of keys
    that went through the rotation.
    """
    g = rng(DATA_SEED, 2, row)
    k = g.standard_normal((past, wl.num_kv_heads, wl.head_dim), dtype=np.float32)
    v = g.standard_normal((past, wl.num_kv_heads, wl.head_dim), dtype=np.float32)
    return k, v


def kv_bytes_read(wl: Workload, total_lengths) -> int:
    """K+V bytes attention must read: sum_b L_b * 2 * Hkv * D * elem_bytes."""
    return int(np.sum(total_lengths)) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def pow2_ge(n: int) -> int:
    return 1 << max(0, math.ceil(math.log2(max(1, n))))
