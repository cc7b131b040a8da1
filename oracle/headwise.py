"""Oracle for headwise mixed 2/4-bit KV precision (TEST INFRASTRUCTURE ONLY).

TurboAttention (arXiv 2412.08585), §3.2 (headwise mixed precision): each
head of a layer gets a priority from two statistics of its values, the
gap^(h) (the difference between the largest and the smallest value over all
of the head's channels) and std^(h) (the standard deviation of the head's
channel-wise gaps); the n_h heads of lowest priority are stored at 2 bits,
the others at 4 bits.  The equation that combines the two statistics is
missing from the page; both are described as "larger means more sensitive",
and the plainest reading that keeps both is their product:

    mx_j, mn_j   = max and min over the head's rows of channel j
    gap_j        = mx_j - mn_j                        (channel-wise gap)
    gap          = max_j mx_j - min_j mn_j
    std          = sqrt(mean_j (gap_j - mean_j gap_j)^2)   (population std)
    priority     = gap * std

Further readings (the page is silent on them):
  * the rows are a prompt's keys or values of one kv-head over every token of
    every sequence in the batch (tokens t < lens[b]); one ranking per layer,
    shared by all sequences, so one cache layout serves the whole batch;
  * a kv-head's keys and values share one bit width, so its priority is the
    larger of its key priority and its value priority;
  * ties in priority go to the lower head index first (the lowest-priority
    n_h heads are the first n_h of a stable ascending sort);
  * a head with no rows has priority 0;
  * the 2-bit and 4-bit codecs are ``oracle.codec2`` and ``oracle.codec``.

Arithmetic: every statistic is binary64, the sums taken in channel order
j = 0, 1, ..., D - 1 with no fused multiply-add, so that an implementation
that follows the same order reproduces the priorities bit for bit and the
ranking (an integer decision) cannot depend on rounding.
"""

from __future__ import annotations

import math

import numpy as np

from . import attention as att
from . import codec
from . import codec2


def head_priority(rows) -> float:
    """priority = gap * std of one head's rows [n, D] (binary32 values)."""
    x = np.asarray(rows, dtype=np.float32)
    if x.shape[0] == 0:
        return 0.0
    mx = x.max(axis=0).astype(np.float64)
    mn = x.min(axis=0).astype(np.float64)
    d = x.shape[1]
    gaps = [float(mx[j]) - float(mn[j]) for j in range(d)]
    gap = float(mx.max()) - float(mn.min())
    total = 0.0
    for g in gaps:
        total += g
    mean = total / d
    sq = 0.0
    for g in gaps:
        e = g - mean
        sq += e * e
    return gap * math.sqrt(sq / d)


def priorities(k, v, lens=None) -> np.ndarray:
    """Per kv-head priority (binary64 [Hkv]) of prompt rows k, v [B, Hkv, n, D]."""
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    B, H, n, _ = k.shape
    ln = [n] * B if lens is None else [max(0, min(int(x), n)) for x in lens]
    out = np.zeros(H, dtype=np.float64)
    for h in range(H):
        kr = np.concatenate([k[b, h, :ln[b]] for b in range(B)])
        vr = np.concatenate([v[b, h, :ln[b]] for b in range(B)])
        out[h] = max(head_priority(kr), head_priority(vr))
    return out


def plan_bits(prio, n_low: int) -> np.ndarray:
    """bits[h] = 2 for the n_low lowest-priority heads (stable), else 4."""
    order = np.argsort(np.asarray(prio, dtype=np.float64), kind="stable")
    bits = np.full(len(prio), 4, dtype=np.int32)
    bits[order[:n_low]] = 2
    return bits


def dequantize_mixed(x, bits) -> np.ndarray:
    """Quantize rows x [B, Hkv, n, D] head by head with its bit width; returns x^ (float64)."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.float64)
    for h, b in enumerate(bits):
        if b == 2:
            w, s = codec2.quantize_pack2(x[:, h])
            out[:, h] = codec2.dequantize2(w, s, x.shape[-1])
        else:
            p, s = codec.quantize_pack(x[:, h])
            out[:, h] = codec.dequantize(p, s)
    return out


def attention_mixed(q, k, v, bits, softmax_scale: float, k_lens=None):
    """Decode/prefill attention over a cache whose kv-heads carry `bits`."""
    return att.attention(q, dequantize_mixed(k, bits), dequantize_mixed(v, bits),
                         softmax_scale, False, k_lens)
