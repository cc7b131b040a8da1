"""Oracle for the FlashQ-style decode buffer (TEST INFRASTRUCTURE ONLY).

TurboAttention (arXiv 2412.08585), §3.3 (the decoding buffer): tokens
generated during decoding wait in a buffer of n_b rows (n_b = 64) quantized to
8 bits with one universal scale, outliers beyond that scale's range being
clamped, so that rows already buffered never need re-quantizing; once the
buffer is full its rows are compressed to the cache's low-bit format.  §3.2
(Equation 9, its first stage): 8-bit symmetric quantization.  The page gives
no formula for the universal scale and its Appendix A (the full algorithm) is
not in the text, so this oracle fixes the plainest reading, with the cache's
own codec (``oracle.codec``, per-row symmetric INT4) as the low-bit format:

    R     = running maximum |x^| of the rows already in the INT4 cache of one
            (sequence, kv-head) and tensor (K or V): with the INT4 codec that
            is 7 * max_t s_t (a row's absmax becomes code +-7 unless its scale
            saturated); while R is 0 (an empty or all-zero history) each
            appended row sets R to its own absmax
    u     = fl16(fl32(R / 127))        universal scale (RNE twice; saturating)
    c     = clamp(RNE(x / u), -127, 127)  int8 code; all codes 0 when u == 0
    x~    = c * u                      buffered value
    flush (64 rows buffered): every x~ row goes through the INT4 codec into
          the cache at the next 64 positions; R = max(R, 7 * max s of those
          rows); u is recomputed; the buffer empties
    attention at a step: one softmax over the cached rows (x^ = c4 * s) and
          the buffered rows (x~), as if concatenated

Exactness of the float64 route for the int8 code: x is binary32 and u
binary16, so a tie x / u = k + 1/2 is exact in binary64 and a non-tie lies
far from it (the same argument as for the INT4 codec); ``numpy.rint`` of the
binary64 quotient is RNE of the exact quotient.
"""

from __future__ import annotations

import numpy as np

from . import attention as att
from . import codec

NB = 64        # buffer rows per (sequence, kv-head)
QMAX8 = 127    # largest int8 code magnitude (symmetric, zero point 0)


def universal_scale(r) -> np.ndarray:
    """u = fl16(fl32(R / 127)), saturating at 65504 (float16)."""
    r32 = np.asarray(r, dtype=np.float32)
    u32 = r32 / np.float32(QMAX8)
    with np.errstate(over="ignore"):
        u16 = u32.astype(np.float16)
    return np.where(np.isinf(u16), np.float16(codec.FP16_MAX), u16).astype(np.float16)


def quantize_int8(x, u) -> np.ndarray:
    """int8 codes of rows x (..., D) with per-row universal scales u (...)."""
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    u64 = np.asarray(u, dtype=np.float16).astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(u64 > 0, np.rint(x64 / np.where(u64 > 0, u64, 1.0)), 0.0)
    return np.clip(q, -QMAX8, QMAX8).astype(np.int8)


def dequantize_int8(c, u) -> np.ndarray:
    """x~ = c * u in float64."""
    return np.asarray(c, dtype=np.float64) * np.asarray(u, dtype=np.float16).astype(np.float64)[..., None]


def history_range(scales) -> np.ndarray:
    """R of a cached history: 7 * max_t s_t over the last axis (0 when empty), float32."""
    s = np.asarray(scales, dtype=np.float16).astype(np.float32)
    if s.shape[-1] == 0:
        return np.zeros(s.shape[:-1], dtype=np.float32)
    return (np.float32(codec.QMAX) * s.max(axis=-1)).astype(np.float32)


class BufferedHead:
    """One (sequence, kv-head) and tensor: INT4 history + int8 buffer, step by step."""

    def __init__(self, history):
        """history: float rows (n, D) already in the cache (quantized with the INT4 codec)."""
        h = np.asarray(history, dtype=np.float32)
        self.packed, self.scales = codec.quantize_pack(h)  # (n, D/2) uint8, (n,) float16
        self.r = history_range(self.scales)
        self.u = universal_scale(self.r) if h.shape[0] else np.float16(0)
        self.codes = []  # buffered int8 rows

    def append(self, row):
        """Buffer one new row; returns its int8 codes."""
        row = np.asarray(row, dtype=np.float32)
        if self.r == 0:  # no range yet: this row sets it
            self.r = np.float32(np.max(np.abs(row)))
            self.u = universal_scale(self.r)
        c = quantize_int8(row[None], np.asarray([self.u]))[0]
        self.codes.append(c)
        return c

    def flush(self):
        """Move a full buffer into the INT4 history; returns the new rows' (packed, scales)."""
        assert len(self.codes) == NB
        xt = dequantize_int8(np.stack(self.codes), np.full(NB, self.u, dtype=np.float16))
        p, s = codec.quantize_pack(xt.astype(np.float32))
        self.packed = np.concatenate([self.packed, p])
        self.scales = np.concatenate([self.scales, s])
        self.r = np.float32(max(float(self.r), float(history_range(s))))
        self.u = universal_scale(self.r)
        self.codes = []
        return p, s

    def values(self):
        """All rows the attention sees: dequantized history, then the buffer (float64)."""
        hist = codec.dequantize(self.packed, self.scales)
        if not self.codes:
            return hist
        buf = dequantize_int8(np.stack(self.codes), np.full(len(self.codes), self.u, dtype=np.float16))
        return np.concatenate([hist, buf])


def attention_buffered(q, k_heads, v_heads, scale):
    """Decode attention over history + buffer.

    q: (G, D) query heads of one kv-head; k_heads, v_heads: BufferedHead.
    Returns O (G, D) and lse (G,) in float64 (oracle.attention's definition).
    """
    k = k_heads.values()
    v = v_heads.values()
    o, l = att.attention(np.asarray(q, dtype=np.float64)[None, :, None, :],
                         k[None, None], v[None, None], scale, False)
    return o[0, :, 0], l[0, :, 0]
