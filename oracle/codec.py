"""Oracle for the INT4 KV-cache codec (TEST INFRASTRUCTURE ONLY).

The format
----------
"Quantized Cross-Attention: Extending FlashAttention-3 with In-SRAM
Dequantization", §3.2 (Tile-Level Quantization), stores a KV tile as 4-bit
codes (128 x 128 x 4 bits = 8 KB) plus one FP16 scale per token
(128 x FP16 = 256 B); its §4.1 kernel signature lays the compressed cache out
as [batch, heads, seq_kv, dim * BIT_WIDTH / 32] words with scales per
(batch, head, token, dim / GROUP_SIZE).  TurboAttention (arXiv 2412.08585),
§2.3, defines symmetric quantization as the zero-point-free case of
Q(x) = round(x / s) + z.  The codec here is that symmetric case at 4 bits,
one group per (token, kv-head) row:

    am   = max_i |x_i|                      (exact)
    s32  = fl32(am / 7)                     (IEEE binary32, round-to-nearest-even)
    s    = fl16(s32)                        (IEEE binary16, RNE; +inf saturates to 65504)
    c_i  = clamp(RNE(x_i / s), -7, 7)       (exact quotient; all codes 0 when s == 0)
    x^_i = c_i * s

Readings taken where the pages are silent or garbled (page 1's LUT in §3.1
has eight entries {-3s..4s} indexed by a 4-bit value, which is not a
consistent codec):
  * symmetric range [-7, 7]; code -8 is never produced;
  * GROUP_SIZE = dim, i.e. one scale per (token, kv-head);
  * the scale is rounded twice (fp32 quotient, then fp16), spelled out above;
  * ties in x / s round half to even, decided on the exact quotient;
  * packing: D/2 bytes per row; element 2k in the low nibble of byte k,
    element 2k+1 in the high nibble; nibbles are two's complement.

Exactness of the float64 route: x is a binary32 value and s a binary16 value,
so a genuine tie x / s = k + 1/2 is exactly representable and a non-tie lies
at least 2**-26 away from k + 1/2, far more than one binary64 ulp of the
quotient.  ``numpy.rint`` on the binary64 quotient therefore equals RNE of
the exact quotient (pinned against exact rationals in the tests).
"""

from __future__ import annotations

import numpy as np

QMAX = 7            # largest code magnitude (symmetric INT4, zero point 0)
FP16_MAX = 65504.0  # largest finite binary16 value (scale saturation)


def row_scales(x) -> np.ndarray:
    """Per-row scale s = fl16(fl32(absmax / 7)) as float16, shape x.shape[:-1].

    TurboAttention (arXiv 2412.08585) §2.3: symmetric quantization has zero
    point 0 and a scale set by the range; the range of a symmetric 4-bit code
    is [-7, 7], so the scale is absmax / 7.
    """
    x32 = np.asarray(x, dtype=np.float32)
    am = np.max(np.abs(x32), axis=-1)
    s32 = am / np.float32(QMAX)               # binary32 division, RNE
    with np.errstate(over="ignore"):
        s16 = s32.astype(np.float16)          # RNE to binary16
    return np.where(np.isinf(s16), np.float16(FP16_MAX), s16).astype(np.float16)


def quantize_rows(x):
    """Quantize rows of ``x`` (float32 or float16, [..., D]).

    Returns (codes int8 [..., D] in [-7, 7], scales float16 [...]).
    """
    x32 = np.asarray(x, dtype=np.float32)
    s16 = row_scales(x32)
    s64 = s16.astype(np.float64)[..., None]
    x64 = x32.astype(np.float64)
    safe = np.where(s64 > 0.0, s64, 1.0)
    q = np.where(s64 > 0.0, x64 / safe, 0.0)
    codes = np.clip(np.rint(q), -QMAX, QMAX).astype(np.int8)
    return codes, s16


def pack_nibbles(codes) -> np.ndarray:
    """Pack int8 codes [..., D] into uint8 [..., D/2]: even element low nibble."""
    c = np.asarray(codes, dtype=np.int8)
    if c.shape[-1] % 2:
        raise ValueError("row length must be even")
    lo = c[..., 0::2].astype(np.uint8) & np.uint8(0x0F)
    hi = c[..., 1::2].astype(np.uint8) & np.uint8(0x0F)
    return (lo | (hi << np.uint8(4))).astype(np.uint8)


def unpack_nibbles(packed) -> np.ndarray:
    """Inverse of :func:`pack_nibbles`: uint8 [..., D/2] -> int8 [..., D]."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & np.uint8(0x0F)).astype(np.int16)
    hi = (p >> np.uint8(4)).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)       # two's complement nibble
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def quantize_pack(x):
    """Quantize and pack: returns (packed uint8 [..., D/2], scales float16 [...])."""
    codes, s = quantize_rows(x)
    return pack_nibbles(codes), s


def dequantize(packed, scales) -> np.ndarray:
    """x^ = c * s in float64, [..., D].

    Page 1 §3.1 ("In-SRAM Dequantization") multiplies each 4-bit value by its
    scale; here that product is taken exactly (it is exact in binary32 too:
    an 11-bit scale times a 3-bit code).
    """
    c = unpack_nibbles(packed).astype(np.float64)
    return c * np.asarray(scales, dtype=np.float16).astype(np.float64)[..., None]


def tile_bytes(tokens: int, dim: int) -> tuple[int, int]:
    """(code bytes, scale bytes) for a tile of ``tokens`` rows of ``dim`` values.

    Page 1 §3.2: a 128 x 128 tile is 8 KB of 4-bit codes plus 256 B of FP16
    scales.
    """
    return tokens * dim // 2, tokens * 2
