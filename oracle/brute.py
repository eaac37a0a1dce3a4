"""Brute-force full recomputation without any cache (numpy, fp64, tiny sizes).

TEST INFRASTRUCTURE ONLY.  An independent second statement of the path used to
pin the cached oracle: the cached K/V of a token "never change" once computed,
so attention of the newest token(s) against a cache must equal attention
recomputed from scratch over the whole sequence ("Hand-writing an LLM inference
engine" series opener, section 2.5 on the KV cache; "Nano-vLLM Part 2" page,
section 05).

RoPE is written here as complex multiplication: the adjacent pair
(x[2i], x[2i+1]) is the complex number x[2i] + 1j*x[2i+1], multiplied by
exp(1j * m * theta_i) ("Tokenizer, KV Cache and RoPE" page, section 4).  It
does not reuse the C oracle's rotation.
"""
from __future__ import annotations

import numpy as np


def rope_complex(x: np.ndarray, positions: np.ndarray, base: float = 10000.0) -> np.ndarray:
    """x[..., T, H, D] rotated at positions[T] via complex multiplication."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    theta = base ** (-2.0 * np.arange(D // 2, dtype=np.float64) / D)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]  # [T, D/2]
    z = x[..., 0::2] + 1j * x[..., 1::2]
    z = z * np.exp(1j * ang)[:, None, :]
    out = np.empty_like(x)
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def causal_attention_full(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: slice | None = None,
                          scale: float | None = None) -> np.ndarray:
    """Full causal attention of one sequence.

    q: [N, Hq, D]; k, v: [N, Hkv, D] (already rotated as wanted); query n sees
    keys 0..n.  Query head j uses KV head j // (Hq // Hkv).  Returns [N, Hq, D]
    or the selected rows.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((N, Hq, D))
    mask = np.tril(np.ones((N, N), dtype=bool))
    for j in range(Hq):
        s = (q[:, j, :] @ k[:, j // G, :].T) * scale
        s = np.where(mask, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, j, :] = p @ v[:, j // G, :]
    return out if rows is None else out[rows]
