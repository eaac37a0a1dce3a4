"""Python binding of kvattn, the GB300 (sm_103a) RoPE + KV-cache + attention library.

Argument marshalling only: every step runs in the CUDA kernels of
``libkvattn.so`` (built from ``csrc/`` by ``build()``), reached through the C
ABI declared in ``include/kvattn.h``.  PyTorch supplies device memory and the
current stream.  There is no CPU fallback: importing this package without the
built library raises, and every call raises ``KvattnError`` on a non-OK status.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

LIB_PATH = _build.LIB

F32 = 0
BF16 = 1

STATUS = {
    0: "KVATTN_OK",
    1: "KVATTN_ERR_INVALID_ARG",
    2: "KVATTN_ERR_UNSUPPORTED",
    3: "KVATTN_ERR_OUT_OF_BLOCKS",
    4: "KVATTN_ERR_WORKSPACE_TOO_SMALL",
    5: "KVATTN_ERR_CUDA",
    6: "KVATTN_ERR_TIMEOUT",
    7: "KVATTN_ERR_BAD_INDEX",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

EXPORTED = [
    "kvattn_version", "kvattn_status_string", "kvattn_rope_append", "kvattn_rope_append_strided",
    "kvattn_decode_workspace_size",
    "kvattn_decode_num_splits", "kvattn_decode", "kvattn_decode_static_scratch", "kvattn_prefill_chunk",
    "kvattn_prefill_fp8_workspace_size", "kvattn_prefill_chunk_fp8",
    "kvattn_selftest_wait_timeout", "kvattn_get_device_status",
    "kvattn_allocator_create", "kvattn_allocator_destroy", "kvattn_alloc_blocks", "kvattn_free_blocks",
    "kvattn_share_blocks", "kvattn_claim_blocks", "kvattn_allocator_num_free", "kvattn_allocator_num_failures",
    "kvattn_allocator_refcount", "kvattn_table_grow", "kvattn_table_release",
    "kvattn_layered_cache_bytes", "kvattn_layer_cache", "kvattn_copy_blocks", "kvattn_copy_blocks_layered",
    "kvattn_table_fork", "kvattn_table_prepare_append", "kvattn_rope_append_fp8", "kvattn_decode_fp8",
]


class KvattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = int(code)
        self.name = STATUS.get(self.code, f"status {code}")
        super().__init__(f"{what}: {self.name}")


class Config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("scale", ctypes.c_float)]


class CacheDesc(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32)]


class CacheFP8Desc(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32)]


FP8_PAGE_BYTES = 4224  # one (block, KV head, 16 tokens) page at head_dim 128


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"kvattn CUDA library not built ({LIB_PATH} missing): run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    i32, i64, p, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    cfgp, cachep = ctypes.POINTER(Config), ctypes.POINTER(CacheDesc)
    sig = {
        "kvattn_version": ([], i32),
        "kvattn_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "kvattn_rope_append": ([cfgp, cachep, p, p, p, p, p, p, i32, i32, i32, p], ctypes.c_int),
        "kvattn_rope_append_strided": ([cfgp, cachep, p, i64, p, i64, p, i64, p, p, p, p, i32, i32, i32, p],
                                       ctypes.c_int),
        "kvattn_layered_cache_bytes": ([cfgp, i32, i64, i32], sz),
        "kvattn_layer_cache": ([cfgp, p, i32, i64, i32, i32, cachep], ctypes.c_int),
        "kvattn_copy_blocks": ([cfgp, cachep, p, p, i32, p], ctypes.c_int),
        "kvattn_rope_append_fp8": ([cfgp, ctypes.POINTER(CacheFP8Desc), p, p, p, p, p, p, i32, i32, i32, p],
                                   ctypes.c_int),
        "kvattn_decode_fp8": ([cfgp, ctypes.POINTER(CacheFP8Desc), p, p, i32, p, i32, i32, i32, p, p, sz, p],
                              ctypes.c_int),
        "kvattn_copy_blocks_layered": ([cfgp, p, i32, i64, i32, p, p, i32, p], ctypes.c_int),
        "kvattn_table_fork": ([p, p, p, i32, i32, i32], ctypes.c_int),
        "kvattn_table_prepare_append": ([p, p, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)],
                                        ctypes.c_int),
        "kvattn_decode_workspace_size": ([cfgp, i32, i32, i32], sz),
        "kvattn_decode_num_splits": ([cfgp, i32, i32, i32], i32),
        "kvattn_decode": ([cfgp, cachep, p, p, i32, p, i32, i32, i32, p, p, sz, p], ctypes.c_int),
        "kvattn_decode_static_scratch": ([cfgp, cachep, p, p, i32, p, i32, i32, i32, p, p], ctypes.c_int),
        "kvattn_prefill_chunk": ([cfgp, cachep, p, p, p, p, i32, i32, i32, i32, p, p], ctypes.c_int),
        "kvattn_prefill_fp8_workspace_size": ([cfgp, i32, i32, i32, i64], sz),
        "kvattn_prefill_chunk_fp8": ([cfgp, ctypes.POINTER(CacheFP8Desc), p, p, p, p, i32, i32, i32, i32, i64, p, p,
                                      sz, p], ctypes.c_int),
        "kvattn_get_device_status": ([p, ctypes.POINTER(i32)], ctypes.c_int),
        "kvattn_selftest_wait_timeout": ([i32, p], ctypes.c_int),
        "kvattn_allocator_create": ([i64, ctypes.POINTER(p)], ctypes.c_int),
        "kvattn_allocator_destroy": ([p], None),
        "kvattn_alloc_blocks": ([p, i32, p], ctypes.c_int),
        "kvattn_free_blocks": ([p, p, i32], ctypes.c_int),
        "kvattn_share_blocks": ([p, p, i32], ctypes.c_int),
        "kvattn_claim_blocks": ([p, p, i32], ctypes.c_int),
        "kvattn_allocator_num_free": ([p], i64),
        "kvattn_allocator_num_failures": ([p], i64),
        "kvattn_allocator_refcount": ([p, i32], i32),
        "kvattn_table_grow": ([p, p, i32, i32, i32, i32], ctypes.c_int),
        "kvattn_table_release": ([p, p, i32, i32, i32], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def check(code: int, what: str) -> None:
    if code != 0:
        raise KvattnError(code, what)


def version() -> int:
    return int(lib.kvattn_version())


def status_string(code: int) -> str:
    return lib.kvattn_status_string(int(code)).decode()


# ------------------------------------------------------------------ torch-facing helpers

def _torch():
    import torch

    return torch


def make_config(num_q_heads: int, num_kv_heads: int, head_dim: int, dtype: int,
                rope_base: float = 10000.0, scale: float = 0.0) -> Config:
    return Config(num_q_heads, num_kv_heads, head_dim, dtype, rope_base, scale)


def dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported element type {t.dtype}")


def _dev(t, name: str, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Cache:
    """One layer's K and V pools, [num_blocks, Hkv, block_size, D] each (device tensors, caller-owned)."""

    def __init__(self, k_pool, v_pool):
        if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
            raise ValueError("k_pool and v_pool must both be [num_blocks, Hkv, block_size, D]")
        self.k_pool, self.v_pool = k_pool, v_pool
        self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = k_pool.shape
        self.desc = CacheDesc(_dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
                              int(self.num_blocks), int(self.block_size))

    @classmethod
    def empty(cls, num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int, dtype, device="cuda"):
        torch = _torch()
        k = torch.empty((num_blocks, num_kv_heads, block_size, head_dim), dtype=dtype, device=device)
        v = torch.empty_like(k)
        return cls(k, v)


class CacheFP8:
    """One layer's fp8 (e4m3) KV cache: a uint8 pool [num_blocks, Hkv,
    block_size // 16, 4224] of pages holding 16 tokens' K codes (chunks
    rotated per row), V codes (transposed) and their per-(slot, head) fp32
    scales; the byte layout is stated in kvattn.h (kvattn_cache_fp8)."""

    def __init__(self, pool, block_size: int = 16):
        torch = _torch()
        if pool.dim() != 4 or pool.dtype != torch.uint8 or pool.shape[3] != FP8_PAGE_BYTES:
            raise ValueError("pool must be uint8 [num_blocks, Hkv, block_size // 16, 4224]")
        if block_size % 16 or pool.shape[2] != block_size // 16:
            raise ValueError("block_size must be a multiple of 16 matching the pool's page count")
        self.pool = pool
        self.num_blocks, self.num_kv_heads = int(pool.shape[0]), int(pool.shape[1])
        self.block_size, self.head_dim = int(block_size), 128
        self.desc = CacheFP8Desc(_dev(pool, "pool"), self.num_blocks, self.block_size)

    @classmethod
    def empty(cls, num_blocks: int, num_kv_heads: int, block_size: int = 16, device="cuda"):
        torch = _torch()
        pool = torch.empty((num_blocks, num_kv_heads, block_size // 16, FP8_PAGE_BYTES), dtype=torch.uint8,
                           device=device)
        return cls(pool, block_size)


def rope_append_fp8(cfg: Config, cache: CacheFP8, q, k, v, positions, seq_ids, block_table, stream=None) -> None:
    """kvattn_rope_append_fp8: rotate bf16 q in place, store rotated k and v as e4m3 rows with scales."""
    torch = _torch()
    check(lib.kvattn_rope_append_fp8(ctypes.byref(cfg), ctypes.byref(cache.desc), _dev(q, "q", torch.bfloat16),
                                     _dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16),
                                     _dev(positions, "positions", torch.int32), _dev(seq_ids, "seq_ids", torch.int32),
                                     _dev(block_table, "block_table", torch.int32), block_table.shape[0],
                                     block_table.shape[1], q.shape[0], _stream(stream)),
          "kvattn_rope_append_fp8")


def decode_fp8(cfg: Config, cache: CacheFP8, q, block_table, seq_lens, max_seq_len: int, out=None,
               workspace=None, num_splits: int = 0, stream=None):
    """kvattn_decode_fp8: decode attention over an fp8 cache (bf16 q and output)."""
    torch = _torch()
    B = q.shape[0]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        n = decode_workspace_size(cfg, B, max_seq_len, num_splits)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    check(lib.kvattn_decode_fp8(ctypes.byref(cfg), ctypes.byref(cache.desc), _dev(q, "q", torch.bfloat16),
                                _dev(block_table, "block_table", torch.int32), block_table.shape[1],
                                _dev(seq_lens, "seq_lens", torch.int32), B, int(max_seq_len), int(num_splits),
                                _dev(out, "out", torch.bfloat16), _dev(workspace, "workspace"), workspace.numel(),
                                _stream(stream)),
          "kvattn_decode_fp8")
    return out


class LayeredCache:
    """Every layer's K and V pools in one device allocation,
    [num_layers, 2, num_blocks, Hkv, block_size, D]: one block id (one block
    table, one allocator) names the same block in all 2 * num_layers regions.
    layer(l) is that layer's Cache, placed by kvattn_layer_cache."""

    def __init__(self, cfg: Config, pool):
        if pool.dim() != 6 or pool.shape[1] != 2:
            raise ValueError("pool must be [num_layers, 2, num_blocks, Hkv, block_size, D]")
        L, _, nb, hkv, bs, d = pool.shape
        if (hkv, d) != (cfg.num_kv_heads, cfg.head_dim):
            raise ValueError("pool heads / head_dim do not match the config")
        _dev(pool, "pool")
        need = int(lib.kvattn_layered_cache_bytes(ctypes.byref(cfg), L, nb, bs))
        if need != pool.numel() * pool.element_size():
            raise ValueError(f"pool holds {pool.numel() * pool.element_size()} bytes, the layout needs {need}")
        self.cfg, self.pool = cfg, pool
        self.num_layers, self.num_blocks, self.block_size = int(L), int(nb), int(bs)

    @classmethod
    def empty(cls, cfg: Config, num_layers: int, num_blocks: int, block_size: int, dtype, device="cuda"):
        torch = _torch()
        pool = torch.empty((num_layers, 2, num_blocks, cfg.num_kv_heads, block_size, cfg.head_dim),
                           dtype=dtype, device=device)
        return cls(cfg, pool)

    def layer(self, l: int) -> "Cache":
        desc = CacheDesc()
        check(lib.kvattn_layer_cache(ctypes.byref(self.cfg), ctypes.c_void_p(self.pool.data_ptr()),
                                     self.num_layers, self.num_blocks, self.block_size, int(l),
                                     ctypes.byref(desc)), "kvattn_layer_cache")
        c = Cache(self.pool[l, 0], self.pool[l, 1])
        if (c.desc.k_pool, c.desc.v_pool) != (desc.k_pool, desc.v_pool):
            raise RuntimeError("kvattn_layer_cache placed the layer away from the pool's [l, 0] / [l, 1] slices")
        c.desc = desc
        return c


def copy_blocks(cfg: Config, cache, src_ids, dst_ids, stream=None) -> None:
    """kvattn_copy_blocks (a Cache) or kvattn_copy_blocks_layered (a LayeredCache):
    block dst_ids[i] := block src_ids[i] in every K and V region.  The ids are
    int32 device tensors, or sequences that are uploaded first."""
    torch = _torch()
    dev = cache.pool.device if isinstance(cache, LayeredCache) else cache.k_pool.device
    src = src_ids if isinstance(src_ids, torch.Tensor) else torch.tensor(list(src_ids), dtype=torch.int32, device=dev)
    dst = dst_ids if isinstance(dst_ids, torch.Tensor) else torch.tensor(list(dst_ids), dtype=torch.int32, device=dev)
    if src.numel() != dst.numel():
        raise ValueError("src_ids and dst_ids differ in length")
    n = src.numel()
    if n == 0:
        return
    sp, dp = _dev(src, "src_ids", torch.int32), _dev(dst, "dst_ids", torch.int32)
    if isinstance(cache, LayeredCache):
        check(lib.kvattn_copy_blocks_layered(ctypes.byref(cfg), ctypes.c_void_p(cache.pool.data_ptr()),
                                             cache.num_layers, cache.num_blocks, cache.block_size, sp, dp, n,
                                             _stream(stream)), "kvattn_copy_blocks_layered")
    else:
        check(lib.kvattn_copy_blocks(ctypes.byref(cfg), ctypes.byref(cache.desc), sp, dp, n, _stream(stream)),
              "kvattn_copy_blocks")


def _rows(t, name: str, heads: int, head_dim: int, dtype=None):
    """Pointer and row stride (elements) of a [T, heads, D] or [T, heads*D] view
    whose rows are dense but may sit at any stride (a slice of a fused QKV row)."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    row = heads * head_dim
    if t.dim() == 3 and tuple(t.shape[1:]) == (heads, head_dim):
        dense = t.shape[2] <= 1 or t.stride(2) == 1
        dense = dense and (t.shape[1] <= 1 or t.stride(1) == head_dim)
    elif t.dim() == 2 and t.shape[1] == row:
        dense = t.shape[1] <= 1 or t.stride(1) == 1
    else:
        raise ValueError(f"{name} must be [T, {heads}, {head_dim}] or [T, {row}]")
    if not dense:
        raise ValueError(f"{name}: each token's row must be dense (heads and dims contiguous)")
    stride = t.stride(0) if t.shape[0] > 1 else row
    return ctypes.c_void_p(t.data_ptr()), int(stride)


def split_qkv(qkv, num_q_heads: int, num_kv_heads: int, head_dim: int):
    """Views q [T,Hq,D], k [T,Hkv,D], v [T,Hkv,D] of one fused QKV projection
    output [T, (Hq + 2 Hkv) D] (no copy); pass them to rope_append as they are."""
    T = qkv.shape[0]
    hq, hkv, d = num_q_heads, num_kv_heads, head_dim
    if qkv.dim() != 2 or qkv.shape[1] != (hq + 2 * hkv) * d:
        raise ValueError(f"qkv must be [T, {(hq + 2 * hkv) * d}]")
    if qkv.stride(1) != 1:
        raise ValueError("qkv rows must be dense")
    q = qkv[:, : hq * d].view(T, hq, d)
    k = qkv[:, hq * d: (hq + hkv) * d].view(T, hkv, d)
    v = qkv[:, (hq + hkv) * d:].view(T, hkv, d)
    return q, k, v


def rope_append(cfg: Config, cache: Cache, q, k, v, positions, seq_ids, block_table, stream=None,
                q_out=None) -> None:
    """kvattn_rope_append: rotate q in place (or into q_out), write rotated k and
    raw v into the cache.

    q, k, v are dense [T, H, D] tensors, or row-strided views (split_qkv of a
    fused QKV output); those, or a q_out, go through kvattn_rope_append_strided."""
    torch = _torch()
    T = q.shape[0]
    hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    common = (_dev(positions, "positions", torch.int32), _dev(seq_ids, "seq_ids", torch.int32),
              _dev(block_table, "block_table", torch.int32),
              block_table.shape[0], block_table.shape[1], T, _stream(stream))
    if q_out is None and q.is_contiguous() and k.is_contiguous() and v.is_contiguous():
        check(lib.kvattn_rope_append(ctypes.byref(cfg), ctypes.byref(cache.desc), _dev(q, "q"),
                                     _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), *common),
              "kvattn_rope_append")
        return
    qp, qs = _rows(q, "q", hq, d)
    kp, ks = _rows(k, "k", hkv, d, q.dtype)
    vp, vs = _rows(v, "v", hkv, d, q.dtype)
    qo = None
    if q_out is not None:
        if tuple(q_out.shape) != (T, hq, d):
            raise ValueError(f"q_out must be [{T}, {hq}, {d}]")
        qo = _dev(q_out, "q_out", q.dtype)
    check(lib.kvattn_rope_append_strided(ctypes.byref(cfg), ctypes.byref(cache.desc), qp, qs, kp, ks, vp, vs,
                                         qo, *common),
          "kvattn_rope_append_strided")


def decode_workspace_size(cfg: Config, batch: int, max_seq_len: int, num_splits: int = 0) -> int:
    return int(lib.kvattn_decode_workspace_size(ctypes.byref(cfg), batch, max_seq_len, num_splits))


def decode_num_splits(cfg: Config, batch: int, max_seq_len: int, num_splits: int = 0) -> int:
    return int(lib.kvattn_decode_num_splits(ctypes.byref(cfg), batch, max_seq_len, num_splits))


def decode(cfg: Config, cache: Cache, q, block_table, seq_lens, max_seq_len: int, out=None,
           workspace=None, num_splits: int = 0, stream=None):
    """kvattn_decode: one query token per sequence against its whole cache."""
    torch = _torch()
    B = q.shape[0]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        n = decode_workspace_size(cfg, B, max_seq_len, num_splits)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    check(lib.kvattn_decode(ctypes.byref(cfg), ctypes.byref(cache.desc), _dev(q, "q"),
                            _dev(block_table, "block_table", torch.int32), block_table.shape[1],
                            _dev(seq_lens, "seq_lens", torch.int32), B, int(max_seq_len), int(num_splits),
                            _dev(out, "out", q.dtype), _dev(workspace, "workspace"), workspace.numel(),
                            _stream(stream)),
          "kvattn_decode")
    return out


def prefill_chunk(cfg: Config, cache: Cache, q, cu_q_lens, prefix_lens, block_table, max_q_len: int,
                  out=None, stream=None):
    """kvattn_prefill_chunk: causal attention of query chunks over their caches."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    check(lib.kvattn_prefill_chunk(ctypes.byref(cfg), ctypes.byref(cache.desc), _dev(q, "q"),
                                   _dev(cu_q_lens, "cu_q_lens", torch.int32),
                                   _dev(prefix_lens, "prefix_lens", torch.int32),
                                   _dev(block_table, "block_table", torch.int32), block_table.shape[1],
                                   prefix_lens.shape[0], int(max_q_len), q.shape[0],
                                   _dev(out, "out", q.dtype), _stream(stream)),
          "kvattn_prefill_chunk")
    return out


def prefill_fp8_workspace_size(cfg: Config, block_size: int, max_blocks_per_seq: int, num_chunks: int,
                               max_kv_tokens: int) -> int:
    """kvattn_prefill_fp8_workspace_size (0 for invalid arguments)."""
    return int(lib.kvattn_prefill_fp8_workspace_size(ctypes.byref(cfg), int(block_size), int(max_blocks_per_seq),
                                                     int(num_chunks), int(max_kv_tokens)))


def prefill_chunk_fp8(cfg: Config, cache: CacheFP8, q, cu_q_lens, prefix_lens, block_table, max_q_len: int,
                      max_kv_tokens: int, out=None, workspace=None, stream=None):
    """kvattn_prefill_chunk_fp8: causal attention of query chunks over an fp8 cache (bf16 q and output)."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    n = prefix_lens.shape[0]
    if workspace is None:
        size = prefill_fp8_workspace_size(cfg, cache.desc.block_size, block_table.shape[1], n, max_kv_tokens)
        workspace = torch.empty(max(size, 256), dtype=torch.uint8, device=q.device)
    check(lib.kvattn_prefill_chunk_fp8(ctypes.byref(cfg), ctypes.byref(cache.desc), _dev(q, "q", torch.bfloat16),
                                       _dev(cu_q_lens, "cu_q_lens", torch.int32),
                                       _dev(prefix_lens, "prefix_lens", torch.int32),
                                       _dev(block_table, "block_table", torch.int32), block_table.shape[1], n,
                                       int(max_q_len), q.shape[0], int(max_kv_tokens),
                                       _dev(out, "out", torch.bfloat16), _dev(workspace, "workspace"),
                                       workspace.numel(), _stream(stream)),
          "kvattn_prefill_chunk_fp8")
    return out


def get_device_status(stream=None) -> int:
    """Waits for the stream and returns (and clears) the device status word."""
    v = ctypes.c_int32(0)
    check(lib.kvattn_get_device_status(_stream(stream), ctypes.byref(v)), "kvattn_get_device_status")
    return int(v.value)


def selftest_wait_timeout(limit_us: int = 1000, stream=None) -> None:
    """Runs the bounded-wait self test (records KVATTN_ERR_TIMEOUT on the device)."""
    check(lib.kvattn_selftest_wait_timeout(int(limit_us), _stream(stream)), "kvattn_selftest_wait_timeout")


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


# ------------------------------------------------------------------ host allocator

class BlockAllocator:
    """Host free list of KV block ids with reference counts (C++, thread-safe)."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        check(lib.kvattn_allocator_create(int(num_blocks), ctypes.byref(h)), "kvattn_allocator_create")
        self._h = h
        self.num_blocks = int(num_blocks)

    def close(self) -> None:
        if self._h:
            lib.kvattn_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int):
        import numpy as np

        out = np.empty(int(n), dtype=np.int32)
        check(lib.kvattn_alloc_blocks(self._h, int(n), out.ctypes.data_as(ctypes.c_void_p)), "kvattn_alloc_blocks")
        return out

    def free(self, ids) -> None:
        import numpy as np

        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        check(lib.kvattn_free_blocks(self._h, a.ctypes.data_as(ctypes.c_void_p), a.size), "kvattn_free_blocks")

    def share(self, ids) -> None:
        import numpy as np

        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        check(lib.kvattn_share_blocks(self._h, a.ctypes.data_as(ctypes.c_void_p), a.size), "kvattn_share_blocks")

    def claim(self, ids) -> None:
        """Takes specific free ids (adopting an existing block table)."""
        import numpy as np

        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        check(lib.kvattn_claim_blocks(self._h, a.ctypes.data_as(ctypes.c_void_p), a.size), "kvattn_claim_blocks")

    def grow(self, table_row, block_size: int, cur_len: int, new_len: int) -> None:
        """Allocates blocks so the int32 numpy row covers new_len tokens (in place)."""
        if table_row.dtype.name != "int32" or not table_row.flags.c_contiguous:
            raise TypeError("table_row must be a contiguous int32 numpy array")
        check(lib.kvattn_table_grow(self._h, table_row.ctypes.data_as(ctypes.c_void_p), table_row.size,
                                    int(block_size), int(cur_len), int(new_len)), "kvattn_table_grow")

    def fork(self, src_row, dst_row, block_size: int, length: int) -> None:
        """Prefix sharing: dst_row takes src_row's blocks covering `length` tokens
        (one more reference each)."""
        for r in (src_row, dst_row):
            if r.dtype.name != "int32" or not r.flags.c_contiguous:
                raise TypeError("table rows must be contiguous int32 numpy arrays")
        if src_row.size != dst_row.size:
            raise ValueError("rows of different widths")
        check(lib.kvattn_table_fork(self._h, src_row.ctypes.data_as(ctypes.c_void_p),
                                    dst_row.ctypes.data_as(ctypes.c_void_p), dst_row.size, int(block_size),
                                    int(length)), "kvattn_table_fork")

    def prepare_append(self, table_row, block_size: int, cur_len: int, new_len: int):
        """Blocks for positions cur_len..new_len-1, with copy on write of a shared
        partial block.  Returns (src, dst) of the block to copy, or None."""
        if table_row.dtype.name != "int32" or not table_row.flags.c_contiguous:
            raise TypeError("table_row must be a contiguous int32 numpy array")
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        check(lib.kvattn_table_prepare_append(self._h, table_row.ctypes.data_as(ctypes.c_void_p), table_row.size,
                                              int(block_size), int(cur_len), int(new_len), ctypes.byref(src),
                                              ctypes.byref(dst)), "kvattn_table_prepare_append")
        return None if src.value < 0 else (src.value, dst.value)

    def release(self, table_row, block_size: int, length: int) -> None:
        if table_row.dtype.name != "int32" or not table_row.flags.c_contiguous:
            raise TypeError("table_row must be a contiguous int32 numpy array")
        check(lib.kvattn_table_release(self._h, table_row.ctypes.data_as(ctypes.c_void_p), table_row.size,
                                       int(block_size), int(length)), "kvattn_table_release")

    @property
    def num_free(self) -> int:
        return int(lib.kvattn_allocator_num_free(self._h))

    @property
    def num_failures(self) -> int:
        return int(lib.kvattn_allocator_num_failures(self._h))

    def refcount(self, block_id: int) -> int:
        return int(lib.kvattn_allocator_refcount(self._h, int(block_id)))
