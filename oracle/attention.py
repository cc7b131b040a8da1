"""Oracle for attention over the dequantized INT4 KV cache (TEST INFRASTRUCTURE ONLY).

The result is defined by TurboAttention (arXiv 2412.08585) §2.2, Equation 2,
computed independently for each head and batch instance:

    S = Q K^T,   P = softmax(S),   H = P V

with the usual softmax scale applied to S.  FlashAttention's tiling and online
softmax (the same section; Milakov & Gimelshein) reach this result exactly up
to rounding order, so the oracle is the plain definition: no tiling, no
online max, no split.  K and V are the dequantized cache (codec.dequantize),
so fusing the dequantization into the attention loop ("Quantized
Cross-Attention ... In-SRAM Dequantization", §3.1) must reproduce this.

Prefill and decode follow TurboAttention §2.1: prefill caches K, V for all
prompt tokens; each decode step appends k_t, v_t and attends q_t against the
whole cache.

Readings taken where the pages are silent:
  * causal masking is bottom-right aligned: query i (of Nq) sees key j (of
    Nk) iff j <= i + Nk - Nq; a single decode query sees every cached key;
  * grouped-query attention maps query head h to kv head h // (Hq / Hkv);
  * the log-sum-exp is the natural logarithm, lse_i = ln sum_j exp(S_ij);
  * a query row that sees no key (empty sequence) gives O = 0, lse = -inf;
  * split-KV partials are (O_c normalised within the chunk, lse_c) and merge
    by O = sum_c exp(lse_c - L) O_c with L = ln sum_c exp(lse_c).
"""

from __future__ import annotations

import numpy as np

from . import codec


def _f64(a) -> np.ndarray:
    return np.asarray(a).astype(np.float64)


def attention(q, k_hat, v_hat, softmax_scale: float, causal: bool = False,
              k_lens=None):
    """Exact attention in float64.

    q      [B, Hq, Nq, D]   (fp16 values are widened exactly)
    k_hat  [B, Hkv, Nk, D]  dequantized keys
    v_hat  [B, Hkv, Nk, D]  dequantized values
    k_lens optional [B] number of valid keys per batch entry (<= Nk)

    Returns (O [B, Hq, Nq, D] float64, lse [B, Hq, Nq] float64).
    """
    q = _f64(q)
    k_hat = _f64(k_hat)
    v_hat = _f64(v_hat)
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k_hat.shape[1], k_hat.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    O = np.zeros((B, Hq, Nq, v_hat.shape[-1]), dtype=np.float64)
    lse = np.full((B, Hq, Nq), -np.inf, dtype=np.float64)
    for b in range(B):
        nk = Nk if k_lens is None else int(k_lens[b])
        if nk == 0:
            continue
        i = np.arange(Nq)[:, None]
        j = np.arange(nk)[None, :]
        visible = (j <= i + nk - Nq) if causal else np.ones((Nq, nk), bool)
        for h in range(Hq):
            kv = h // G
            S = softmax_scale * (q[b, h] @ k_hat[b, kv, :nk].T)      # [Nq, nk]
            S = np.where(visible, S, -np.inf)
            rowmax = S.max(axis=1)
            live = np.isfinite(rowmax)
            if not live.any():
                continue
            E = np.exp(S[live] - rowmax[live, None])
            Z = E.sum(axis=1)
            P = E / Z[:, None]
            O[b, h, live] = P @ v_hat[b, kv, :nk]
            lse[b, h, live] = rowmax[live] + np.log(Z)
    return O, lse


def attention_quantized(q, k_packed, k_scales, v_packed, v_scales,
                        softmax_scale: float, causal: bool = False, k_lens=None):
    """Attention straight from the packed cache: dequantize, then attend."""
    return attention(q, codec.dequantize(k_packed, k_scales),
                     codec.dequantize(v_packed, v_scales),
                     softmax_scale, causal, k_lens)


def gather_pages(pool_packed, pool_scales, page_table, seq_lens, page_size: int):
    """Gather a paged cache into contiguous per-sequence form.

    pool_packed [P, Hkv, page_size, D/2], pool_scales [P, Hkv, page_size],
    page_table [B, max_pages] (int, -1 = unused), seq_lens [B].
    Returns (packed [B, Hkv, Lmax, D/2], scales [B, Hkv, Lmax]) where rows past
    a sequence's length are zero.  Token t of sequence b lives in physical page
    page_table[b, t // page_size] at offset t % page_size.
    """
    pool_packed = np.asarray(pool_packed)
    pool_scales = np.asarray(pool_scales)
    seq_lens = [int(x) for x in np.asarray(seq_lens)]
    B = len(seq_lens)
    Hkv, half = pool_packed.shape[1], pool_packed.shape[3]
    L = max(seq_lens) if B else 0
    out_p = np.zeros((B, Hkv, L, half), dtype=np.uint8)
    out_s = np.zeros((B, Hkv, L), dtype=np.float16)
    for b in range(B):
        for t in range(seq_lens[b]):
            page = int(page_table[b][t // page_size])
            off = t % page_size
            out_p[b, :, t] = pool_packed[page, :, off]
            out_s[b, :, t] = pool_scales[page, :, off]
    return out_p, out_s


def combine(partial_o, partial_lse):
    """Log-sum-exp merge of split partials.

    partial_o [S, ..., D] (each normalised within its chunk),
    partial_lse [S, ...].  Returns (O [..., D], lse [...]).  Chunks with
    lse = -inf (no visible key) carry zero weight; if every chunk is empty the
    result is O = 0, lse = -inf.
    """
    po = _f64(partial_o)
    pl = _f64(partial_lse)
    m = pl.max(axis=0)
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    w = np.where(np.isfinite(pl), np.exp(pl - m_safe[None]), 0.0)
    Z = w.sum(axis=0)
    Zs = np.where(live, Z, 1.0)
    O = np.where(live[..., None], (w[..., None] * po).sum(axis=0) / Zs[..., None], 0.0)
    lse = np.where(live, m_safe + np.log(Zs), -np.inf)
    return O, lse


def split_partials(q, k_hat, v_hat, softmax_scale: float, bounds, k_lens=None):
    """Non-causal attention of q over each key chunk [bounds[c], bounds[c+1]).

    Returns (partial_o [S, B, Hq, Nq, D], partial_lse [S, B, Hq, Nq]) with each
    chunk's output normalised over that chunk alone; keys at or past k_lens[b]
    are excluded.  Used to pin :func:`combine`.
    """
    q = _f64(q)
    k_hat = _f64(k_hat)
    v_hat = _f64(v_hat)
    B, Nk = k_hat.shape[0], k_hat.shape[2]
    lens = [Nk] * B if k_lens is None else [int(x) for x in k_lens]
    parts_o, parts_l = [], []
    for c in range(len(bounds) - 1):
        lo, hi = int(bounds[c]), int(bounds[c + 1])
        sub_lens = [max(0, min(hi, n) - lo) for n in lens]
        w = max(hi - lo, 0)
        kk = np.zeros(k_hat.shape[:2] + (w, k_hat.shape[3]))
        vv = np.zeros(v_hat.shape[:2] + (w, v_hat.shape[3]))
        kk[:, :, : max(0, min(hi, Nk) - lo)] = k_hat[:, :, lo:hi]
        vv[:, :, : max(0, min(hi, Nk) - lo)] = v_hat[:, :, lo:hi]
        o, l = attention(q, kk, vv, softmax_scale, False, sub_lens)
        parts_o.append(o)
        parts_l.append(l)
    return np.stack(parts_o), np.stack(parts_l)
