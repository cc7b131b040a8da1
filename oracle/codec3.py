"""Oracle for the INT3 KV-cache codec (TEST INFRASTRUCTURE ONLY).

"Quantized Cross-Attention: Extending FlashAttention-3 with In-SRAM
Dequantization", §3.3 (split-K dequantization): 3-bit values are packed ten
to a 32-bit integer, value i of a word in bits [3i, 3i + 3).  The page says
nothing else about the format, so this oracle takes the INT4 codec's
readings (``oracle.codec``) at 3 bits, one group per (token, kv-head) row:

    am   = max_i |x_i|                      (exact)
    s    = fl16(fl32(am / 3))               (RNE twice; +inf saturates to 65504)
    c_i  = clamp(RNE(x_i / s), -3, 3)       (exact quotient; all codes 0 when s == 0)
    x^_i = c_i * s

Packing: ceil(D / 10) little-endian 32-bit words per row (13 at D = 128, 52
bytes); element j in word j // 10, bits [3 (j % 10), 3 (j % 10) + 3), as a
3-bit two's-complement field; fields past D and bits 30-31 are zero.  Code -4
is never produced.

Exactness of the float64 route: as for the INT4 codec (x binary32, s
binary16, so a tie x / s = k + 1/2 is exact and a non-tie far from it);
``numpy.rint`` of the binary64 quotient is RNE of the exact quotient.
"""

from __future__ import annotations

import numpy as np

from .codec import FP16_MAX

QMAX3 = 3       # largest code magnitude (symmetric INT3, zero point 0)
PER_WORD = 10   # 3-bit values per 32-bit word


def words_per_row(d: int) -> int:
    return -(-d // PER_WORD)


def row_scales3(x) -> np.ndarray:
    """Per-row scale s = fl16(fl32(absmax / 3)) as float16, shape x.shape[:-1]."""
    x32 = np.asarray(x, dtype=np.float32)
    am = np.max(np.abs(x32), axis=-1)
    s32 = am / np.float32(QMAX3)
    with np.errstate(over="ignore"):
        s16 = s32.astype(np.float16)
    return np.where(np.isinf(s16), np.float16(FP16_MAX), s16).astype(np.float16)


def quantize_rows3(x):
    """Codes int8 [..., D] in [-3, 3] and scales float16 [...]."""
    x32 = np.asarray(x, dtype=np.float32)
    s16 = row_scales3(x32)
    s64 = s16.astype(np.float64)[..., None]
    safe = np.where(s64 > 0.0, s64, 1.0)
    q = np.where(s64 > 0.0, x32.astype(np.float64) / safe, 0.0)
    return np.clip(np.rint(q), -QMAX3, QMAX3).astype(np.int8), s16


def pack10(codes) -> np.ndarray:
    """int8 codes [..., D] -> uint32 words [..., ceil(D / 10)]."""
    c = np.asarray(codes, dtype=np.int64)
    d = c.shape[-1]
    nw = words_per_row(d)
    padded = np.zeros(c.shape[:-1] + (nw * PER_WORD,), dtype=np.int64)
    padded[..., :d] = c & 7                      # 3-bit two's complement field
    fields = padded.reshape(c.shape[:-1] + (nw, PER_WORD))
    shifts = 3 * np.arange(PER_WORD, dtype=np.int64)
    return np.sum(fields << shifts, axis=-1).astype(np.uint32)


def unpack10(words, d: int) -> np.ndarray:
    """Inverse of :func:`pack10`: uint32 [..., W] -> int8 [..., d]."""
    w = np.asarray(words, dtype=np.uint32).astype(np.int64)
    shifts = 3 * np.arange(PER_WORD, dtype=np.int64)
    f = (w[..., None] >> shifts) & 7
    f = np.where(f >= 4, f - 8, f)
    return f.reshape(w.shape[:-1] + (w.shape[-1] * PER_WORD,))[..., :d].astype(np.int8)


def quantize_pack3(x):
    """Returns (packed uint32 words [..., ceil(D/10)], scales float16 [...])."""
    c, s = quantize_rows3(x)
    return pack10(c), s


def dequantize3(words, scales, d: int) -> np.ndarray:
    """x^ = c * s in float64, [..., d]."""
    return unpack10(words, d).astype(np.float64) * np.asarray(scales, dtype=np.float16).astype(np.float64)[..., None]
