"""fp64 CPU oracle for the RoPE + KV-cache append + cached attention path.

TEST INFRASTRUCTURE ONLY.  tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library
(``kv_cache_attention_rope_gb300``) never does, and this package never
imports the library.  The two share nothing but the seeded input generators
in ``workloads.py``, which hold none of the method's arithmetic.

What each function follows (the pages are tutorials on hand-writing an LLM
inference engine):

* ``rope`` -- "Tokenizer, KV Cache and RoPE" page, section 4: adjacent pairs
  (x[2i], x[2i+1]) rotated by m * theta_i, theta_i = base^(-2i/d), m the
  token position.
* ``append`` -- "From-scratch AI inference engine" page, section 3.2 (write the
  new token's K/V at the cache index equal to its position) and "Nano-vLLM
  Part 2" page, section 05 (physical block = table[t // BS], offset t % BS).
* ``attend`` -- "From-scratch AI inference engine" page, sections 3.1 and 3.3:
  softmax(q K^T / sqrt(d_k)) V, scale before softmax, causal visibility of
  keys 0..position.
* ``round_to`` -- round-to-nearest-even of the fp64 value to the stored type
  (a reading: the pages do not state a rounding rule).

The C part (``kvattn_oracle.c``) is compiled with plain gcc on first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvattn_oracle.so")
_lib = None
_lock = threading.Lock()

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no machine-specific flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d, i32, i64, p = ctypes.c_double, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            lib.kvo_round_bf16.argtypes = [d]
            lib.kvo_round_bf16.restype = d
            lib.kvo_round_f32.argtypes = [d]
            lib.kvo_round_f32.restype = d
            lib.kvo_round_array.argtypes = [p, i64, i32, p]
            lib.kvo_round_array.restype = None
            lib.kvo_rope.argtypes = [p, i64, i32, i32, p, d, p]
            lib.kvo_rope.restype = ctypes.c_int
            lib.kvo_append.argtypes = [p, p, i64, i32, i32, p, p, p, i32, i32, i32, i64, p, p]
            lib.kvo_append.restype = ctypes.c_int
            lib.kvo_attend.argtypes = [p, i64, i32, i32, i32, p, p, p, p, p, i32, i32, i64, d, p, i32]
            lib.kvo_attend.restype = ctypes.c_int
            lib.kvo_num_cores.argtypes = []
            lib.kvo_num_cores.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_cores() -> int:
    return int(_load().kvo_num_cores())


def round_to(x, dtype: int) -> np.ndarray:
    """Round-to-nearest-even of fp64 values to bf16 (dtype=1) or fp32 (dtype=0), as fp64."""
    x = _f64(x)
    out = np.empty_like(x)
    _load().kvo_round_array(_ptr(x), x.size, int(dtype), _ptr(out))
    return out


def round_bf16_scalar(x: float) -> float:
    return float(_load().kvo_round_bf16(float(x)))


def rope(x, positions, base: float = 10000.0) -> np.ndarray:
    """Rotate x[T, H, D] (fp64, unrounded result) at positions[T]."""
    x = _f64(x)
    if x.ndim != 3:
        raise ValueError("rope expects [T, H, D]")
    T, H, D = x.shape
    pos = _i32(positions)
    out = np.empty_like(x)
    rc = _load().kvo_rope(_ptr(x), T, H, D, _ptr(pos), float(base), _ptr(out))
    if rc:
        raise ValueError(f"kvo_rope failed ({rc})")
    return out


class Cache:
    """The oracle's own KV cache: slot-major Kc[num_blocks*BS, Hkv, D] in fp64."""

    def __init__(self, num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                 fill: float = np.nan):
        self.num_blocks, self.BS = int(num_blocks), int(block_size)
        self.Hkv, self.D = int(num_kv_heads), int(head_dim)
        n = self.num_blocks * self.BS
        self.K = np.full((n, self.Hkv, self.D), fill, dtype=np.float64)
        self.V = np.full((n, self.Hkv, self.D), fill, dtype=np.float64)


def append(cache: Cache, k_rows, v_rows, positions, seq_ids, block_table) -> None:
    """Write already-rotated-and-rounded k_rows[T,Hkv,D] and v_rows into the cache."""
    k, v = _f64(k_rows), _f64(v_rows)
    pos, sid, tab = _i32(positions), _i32(seq_ids), _i32(block_table)
    if tab.ndim != 2:
        raise ValueError("block_table must be [rows, max_blocks]")
    T = k.shape[0]
    rc = _load().kvo_append(_ptr(k), _ptr(v), T, cache.Hkv, cache.D, _ptr(pos), _ptr(sid), _ptr(tab),
                            tab.shape[0], tab.shape[1], cache.BS, cache.num_blocks,
                            _ptr(cache.K), _ptr(cache.V))
    if rc:
        raise IndexError(f"kvo_append failed ({rc})")


def attend(cache: Cache, q, q_rows, q_pos, block_table, num_q_heads: int,
           scale: float | None = None, nthreads: int = 0) -> np.ndarray:
    """Causal attention of q[NQ, Hq, D] (query n sees keys 0..q_pos[n] of row q_rows[n])."""
    qa = _f64(q)
    NQ, Hq, D = qa.shape
    if Hq != num_q_heads or D != cache.D:
        raise ValueError("shape mismatch")
    rows, pos, tab = _i32(q_rows), _i32(q_pos), _i32(block_table)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((NQ, Hq, D), dtype=np.float64)
    rc = _load().kvo_attend(_ptr(qa), NQ, Hq, cache.Hkv, D, _ptr(rows), _ptr(pos), _ptr(cache.K),
                            _ptr(cache.V), _ptr(tab), tab.shape[1], cache.BS, cache.num_blocks,
                            float(scale), _ptr(out), int(nthreads))
    if rc:
        raise IndexError(f"kvo_attend failed ({rc})")
    return out
