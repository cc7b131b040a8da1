"""Oracle for progressive INT8 -> INT4 KV storage (TEST INFRASTRUCTURE ONLY).

TurboAttention (arXiv 2412.08585), §3.1 (Blockwise Progressive
Quantization) and §2.3 (progressive quantization, after QServe): each
FlashAttention sub-block of K or V (the rows of one head in one tile along the
tokens) is first quantized with 8-bit symmetric quantization, one FP16 scale
per sub-block; for storage the 8-bit tensor is then compressed to INT4 with
asymmetric quantization along each channel ("groups in each channel of the key
and value 8-bit tensors"), whose integer scale and zero point are kept in INT8
while the data is kept in INT4; reading it back is dequantization from INT4 to
INT8 (integer scale and zero point), then by the FP16 scale.  §3.3: the
decode buffer's 64 rows, already 8-bit with one universal scale, are
compressed this way once the buffer is full.

The page's equations are missing from the text; the plainest reading of the
prose is taken and written out here (every step exact):

    block      T = 64 consecutive tokens of one (sequence, kv-head) and tensor
    stage 1    s1 = fl16(fl32(absmax(block) / 127)) (RNE twice, saturating),
               q1 = clamp(RNE(x / s1), -127, 127), all 0 when s1 == 0
               (oracle.flashq's int8 code with the block's range); for a full
               decode buffer, q1 and s1 are the buffer's own codes and u
    stage 2    per channel d of the block: lo = min_t q1, hi = max_t q1,
               s2 = max(1, ceil((hi - lo) / 15)) (an integer, 1..17),
               z2 = lo (an int8), q2 = RNE((q1 - lo) / s2) on the exact
               rational (ties to even), in [0, 15] (the ceiling keeps it there)
    storage    q2 as unsigned nibbles, D/2 bytes per token (element 2k in the
               low nibble of byte k); s2 (uint8) and z2 (int8) per block and
               channel; s1 (fp16) per block
    read       q1' = q2 * s2 + z2 (an integer, |q1'| <= 127 + s2 / 2),
               x^ = q1' * s1 (exact in binary64)

Attention over such a cache is attention.attention on x^.
"""

from __future__ import annotations

import numpy as np

from . import attention as att
from . import flashq

BLOCK = 64      # tokens per block (a FlashAttention sub-block; the decode buffer's rows)
QMAX4 = 15      # largest unsigned 4-bit code


def stage1(x):
    """Symmetric 8-bit codes of one block x (T, D): (q1 int8 (T, D), s1 float16)."""
    x32 = np.asarray(x, dtype=np.float32)
    s1 = flashq.universal_scale(np.max(np.abs(x32)) if x32.size else np.float32(0))
    return flashq.quantize_int8(x32, np.broadcast_to(s1, x32.shape[:-1])), np.float16(s1)


def stage2(q1):
    """Channel-wise asymmetric 4-bit codes of int8 codes q1 (T, D):
    (q2 uint8 (T, D) in 0..15, s2 uint8 (D,), z2 int8 (D,))."""
    q = np.asarray(q1, dtype=np.int64)
    lo, hi = q.min(axis=0), q.max(axis=0)
    s2 = np.maximum(1, -((lo - hi) // QMAX4))           # ceil((hi - lo) / 15), at least 1
    num = q - lo                                          # 0 .. hi - lo, exact
    # RNE(num / s2) with exact integer arithmetic: floor, then the half-way rule
    fl, rem = num // s2, num % s2
    up = (2 * rem > s2) | ((2 * rem == s2) & (fl % 2 == 1))
    q2 = np.clip(fl + up, 0, QMAX4)
    return q2.astype(np.uint8), s2.astype(np.uint8), lo.astype(np.int8)


def pack_unsigned(q2) -> np.ndarray:
    """(..., D) codes 0..15 -> (..., D/2) bytes, element 2k in the low nibble."""
    q = np.asarray(q2, dtype=np.uint8)
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def unpack_unsigned(packed) -> np.ndarray:
    """Inverse of pack_unsigned."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def read_int8(q2, s2, z2) -> np.ndarray:
    """q1' = q2 * s2 + z2 (int64), broadcasting the per-channel s2, z2."""
    return np.asarray(q2, dtype=np.int64) * np.asarray(s2, dtype=np.int64) + np.asarray(z2, dtype=np.int64)


def quantize_blocks(x):
    """x (..., N, D) float, N a multiple of 64 -> (packed (..., N, D/2) uint8,
    s1 (..., N/64) float16, s2 (..., N/64, D) uint8, z2 (..., N/64, D) int8)."""
    x = np.asarray(x, dtype=np.float32)
    *lead, N, D = x.shape
    if N % BLOCK:
        raise ValueError("N must be a multiple of 64")
    nb = N // BLOCK
    xb = x.reshape(-1, nb, BLOCK, D)
    packed = np.empty((xb.shape[0], nb, BLOCK, D // 2), np.uint8)
    s1 = np.empty((xb.shape[0], nb), np.float16)
    s2 = np.empty((xb.shape[0], nb, D), np.uint8)
    z2 = np.empty((xb.shape[0], nb, D), np.int8)
    for i in range(xb.shape[0]):
        for j in range(nb):
            q1, s = stage1(xb[i, j])
            q2, a, z = stage2(q1)
            packed[i, j], s1[i, j], s2[i, j], z2[i, j] = pack_unsigned(q2), s, a, z
    return (packed.reshape(*lead, N, D // 2), s1.reshape(*lead, nb), s2.reshape(*lead, nb, D),
            z2.reshape(*lead, nb, D))


def compress_int8_block(q1, s1):
    """A full decode buffer (int8 codes q1 (64, D), universal scale s1) as one
    stored block: (packed (64, D/2), s1, s2 (D,), z2 (D,))."""
    q2, s2, z2 = stage2(q1)
    return pack_unsigned(q2), np.float16(s1), s2, z2


def dequantize_blocks(packed, s1, s2, z2) -> np.ndarray:
    """x^ (..., N, D) in float64 from quantize_blocks' outputs."""
    q2 = unpack_unsigned(packed)
    *lead, N, D = q2.shape
    nb = N // BLOCK
    qb = q2.reshape(*lead, nb, BLOCK, D)
    q1 = read_int8(qb, np.asarray(s2)[..., None, :], np.asarray(z2)[..., None, :])
    x = q1.astype(np.float64) * np.asarray(s1, dtype=np.float16).astype(np.float64)[..., None, None]
    return x.reshape(*lead, N, D)


def attention_pq(q, k_store, v_store, softmax_scale: float, causal: bool = False, k_lens=None):
    """Attention over a stored cache: k_store, v_store = quantize_blocks' tuples."""
    return att.attention(q, dequantize_blocks(*k_store), dequantize_blocks(*v_store), softmax_scale, causal, k_lens)
