"""Oracle for the comparison paths of the fused kernel (TEST INFRASTRUCTURE ONLY).

"Quantized Cross-Attention: Extending FlashAttention-3 with In-SRAM
Dequantization", §5.2 (Baselines) and §5.3 (Results), measures the fused
4-bit kernel against two other ways of computing the same attention:

  * an FP16 FlashAttention-3 kernel, whose K and V are stored in FP16;
  * "post-dequantization": the 4-bit cache is first dequantized into an FP16
    copy in HBM, and that copy is then attended by the FP16 kernel.

Both are defined here as plainly as the fused path is in attention.py:

    fp16 attention          attention(q, K16, V16) on the FP16 values, exactly
    dequantize to FP16      x16_i = fl16(c_i * s)      (IEEE binary16, RNE)
    post-dequantization     attention(q, fl16(c * s_K), fl16(c * s_V))

Reading taken where the page is silent: the FP16 copy is the binary16
rounding (round to nearest, ties to even) of the exact product c * s; the
product is exact in binary32 (an 11-bit scale times a 3-bit code), so a
kernel that multiplies in fp32 and rounds once to fp16 reaches these bits.
A product beyond the binary16 range (only possible for a scale saturated at
65504 and |c| >= 2) becomes +-inf, as IEEE rounding gives.
"""

from __future__ import annotations

import numpy as np

from . import attention as att
from . import codec


def dequantize_fp16(packed, scales) -> np.ndarray:
    """x16 = fl16(c * s) as float16, [..., D]: the FP16 copy a dequantize-first
    path writes to HBM (Quantized Cross-Attention §5.2, post-dequantization)."""
    exact = codec.dequantize(packed, scales)          # c * s, exact in float64
    with np.errstate(over="ignore"):
        return exact.astype(np.float16)               # one RNE rounding to binary16


def attention_fp16(q, k16, v16, softmax_scale: float, causal: bool = False, k_lens=None):
    """Attention over an FP16 KV cache (the FP16 baseline of §5.2): the plain
    definition of attention.attention on the FP16 values, in float64."""
    return att.attention(q, np.asarray(k16, dtype=np.float16), np.asarray(v16, dtype=np.float16),
                         softmax_scale, causal, k_lens)


def attention_post_dequant(q, k_packed, k_scales, v_packed, v_scales, softmax_scale: float,
                           causal: bool = False, k_lens=None):
    """The post-dequantization path: the cache dequantized to FP16, then attended."""
    return attention_fp16(q, dequantize_fp16(k_packed, k_scales), dequantize_fp16(v_packed, v_scales),
                          softmax_scale, causal, k_lens)
