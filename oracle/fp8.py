"""e4m3 (fp8) quantisation of KV-cache rows, for the fp64 oracle.

TEST INFRASTRUCTURE ONLY, like the rest of this package: tests/, smoke() and
the CPU-baseline leg of bench.py may import it; the library never does.

What it follows.  "Tokenizer, KV Cache and RoPE" page, section 2: besides
growing with new tokens and being shared across requests, the KV cache has to
support precision compression, 16-bit values quantised to 8 bits.  The pages
name no format or scaling rule, so this module fixes the reading the library
documents (include/kvattn.h, kvattn_rope_append_fp8):

* format e4m3: sign bit, 4 exponent bits with bias 7, 3 mantissa bits; an
  exponent field of 0 holds the subnormals m/8 * 2^-6; S.1111.111 is NaN;
  there are no infinities; the largest finite magnitude is 1.75 * 2^8 = 448;
* one scale per (slot, KV head) row of D values r (the stored bf16 values):
  amax = max |r|, scale = fp32(amax / 448), inv = fp32(448 / amax) (both 1
  for an all-zero row), code = e4m3(fp32(r * inv)) rounded to nearest, ties
  to the even mantissa, magnitudes past 448 saturated to 448;
* dequantised value = code * scale.

Every step is the definition written out: fp32 operations are numpy float32
operations (IEEE, round to nearest even), the e4m3 rounding is done in fp64
where it is exact (scaling by powers of two, integer rounding).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8), as fp64; NaN for the NaN patterns."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """e4m3 code of each finite value: round to nearest even, saturate at 448."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("e4m3_encode takes finite values")
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))     # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    e = np.clip(ex - 1, -6, 8)                      # binade; below 2^-6 the subnormal spacing 2^-9
    q = np.exp2(e - 3.0)                            # grid spacing in that binade
    v = np.rint(a / q) * q                          # exact scaling; rint: ties to even
    v = np.minimum(v, E4M3_MAX)
    # bits of the grid value v
    _, ev = np.frexp(np.where(v > 0, v, 1.0))
    ev = ev - 1
    normal = v >= 2.0 ** -6
    mant = np.where(normal, v / np.exp2(ev.astype(np.float64)) - 1.0, 0.0) * 8.0
    bits_n = ((ev + 7) << 3) + np.rint(mant).astype(np.int64)
    bits_s = np.rint(v / 2.0 ** -9).astype(np.int64)
    bits = np.where(normal, bits_n, bits_s)
    bits = bits | np.where(np.signbit(x), 0x80, 0)
    return bits.astype(np.uint8)


def quantize_rows(r):
    """Codes [..., D] (uint8) and scales [...] (float32) of rows r [..., D] of
    fp32-representable values (the stored bf16 values of k or v)."""
    r32 = np.asarray(r, dtype=np.float64).astype(np.float32)
    if not np.array_equal(r32.astype(np.float64), np.asarray(r, dtype=np.float64)):
        raise ValueError("quantize_rows takes fp32-representable values")
    amax = np.max(np.abs(r32), axis=-1)
    pos = amax > 0
    safe = np.where(pos, amax, np.float32(1))
    scale = np.where(pos, safe / np.float32(448.0), np.float32(1)).astype(np.float32)
    inv = np.where(pos, np.float32(448.0) / safe, np.float32(1)).astype(np.float32)
    y = (r32 * inv[..., None]).astype(np.float32)
    return e4m3_encode(y.astype(np.float64)), scale


def dequantize_rows(codes, scale) -> np.ndarray:
    """code * scale in fp64."""
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]
