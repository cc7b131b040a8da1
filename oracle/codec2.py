"""Oracle for the INT2 KV-cache codec (TEST INFRASTRUCTURE ONLY).

TurboAttention (arXiv 2412.08585), §3.2 (headwise mixed precision), sends the
lowest-priority heads of a layer to 2-bit and keeps the rest at 4-bit.  Its
own 2-bit format is the asymmetric, channel-wise second stage of its
progressive quantization (§3.1), whose equations the page does not print.
This library stores every bit width in the same per-row symmetric layout
(``oracle.codec`` at 4 bits, ``oracle.codec3`` at 3), so the reading taken
here is that codec at 2 bits, one group per (token, kv-head) row:

    am   = max_i |x_i|                      (exact)
    s    = fl16(fl32(am / 1))               (= fl16(am); +inf saturates to 65504)
    c_i  = clamp(RNE(x_i / s), -1, 1)       (exact quotient; all codes 0 when s == 0)
    x^_i = c_i * s

A symmetric 2-bit code with zero point 0 has three levels {-s, 0, s}; code
-2 is never produced.  A tie |x_i| / s = 1/2 rounds to 0 (half to even).

Packing: D / 16 little-endian 32-bit words per row (8 at D = 128, 32 bytes);
element j in word j // 16, bits [2 (j % 16), 2 (j % 16) + 2), as a 2-bit
two's-complement field (-1 -> 0b11, 0 -> 0b00, 1 -> 0b01).

Exactness of the float64 route: as for the INT4 codec (x binary32, s
binary16, so a tie x / s = k + 1/2 is exact and a non-tie far from it);
``numpy.rint`` of the binary64 quotient is RNE of the exact quotient.
"""

from __future__ import annotations

import numpy as np

from .codec import FP16_MAX

QMAX2 = 1       # largest code magnitude (symmetric INT2, zero point 0)
PER_WORD = 16   # 2-bit values per 32-bit word


def words_per_row(d: int) -> int:
    return -(-d // PER_WORD)


def row_scales2(x) -> np.ndarray:
    """Per-row scale s = fl16(fl32(absmax / 1)) as float16, shape x.shape[:-1]."""
    x32 = np.asarray(x, dtype=np.float32)
    am = np.max(np.abs(x32), axis=-1)
    s32 = am / np.float32(QMAX2)
    with np.errstate(over="ignore"):
        s16 = s32.astype(np.float16)
    return np.where(np.isinf(s16), np.float16(FP16_MAX), s16).astype(np.float16)


def quantize_rows2(x):
    """Codes int8 [..., D] in [-1, 1] and scales float16 [...]."""
    x32 = np.asarray(x, dtype=np.float32)
    s16 = row_scales2(x32)
    s64 = s16.astype(np.float64)[..., None]
    safe = np.where(s64 > 0.0, s64, 1.0)
    q = np.where(s64 > 0.0, x32.astype(np.float64) / safe, 0.0)
    return np.clip(np.rint(q), -QMAX2, QMAX2).astype(np.int8), s16


def pack16(codes) -> np.ndarray:
    """int8 codes [..., D] -> uint32 words [..., ceil(D / 16)]."""
    c = np.asarray(codes, dtype=np.int64)
    d = c.shape[-1]
    nw = words_per_row(d)
    padded = np.zeros(c.shape[:-1] + (nw * PER_WORD,), dtype=np.int64)
    padded[..., :d] = c & 3                      # 2-bit two's complement field
    fields = padded.reshape(c.shape[:-1] + (nw, PER_WORD))
    shifts = 2 * np.arange(PER_WORD, dtype=np.int64)
    return np.sum(fields << shifts, axis=-1).astype(np.uint32)


def unpack16(words, d: int) -> np.ndarray:
    """Inverse of :func:`pack16`: uint32 [..., W] -> int8 [..., d]."""
    w = np.asarray(words, dtype=np.uint32).astype(np.int64)
    shifts = 2 * np.arange(PER_WORD, dtype=np.int64)
    f = (w[..., None] >> shifts) & 3
    f = np.where(f >= 2, f - 4, f)
    return f.reshape(w.shape[:-1] + (w.shape[-1] * PER_WORD,))[..., :d].astype(np.int8)


def quantize_pack2(x):
    """Returns (packed uint32 words [..., ceil(D/16)], scales float16 [...])."""
    c, s = quantize_rows2(x)
    return pack16(c), s


def dequantize2(words, scales, d: int) -> np.ndarray:
    """x^ = c * s in float64, [..., d]."""
    return unpack16(words, d).astype(np.float64) * np.asarray(scales, dtype=np.float16).astype(np.float64)[..., None]
