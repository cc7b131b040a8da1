"""Seeded synthetic inputs shaped like the decode and prefill settings.

This module holds no arithmetic of the method: it only draws random numbers
(and random layouts) from fixed seeds, on the CPU, so the same inputs reach
both the CUDA path and the float64 oracle.  Every (sequence, kv-head) slice
of K or V has its own generator state, so any slice can be regenerated on
its own (the oracle checks sampled slices of full-size workloads that way).

Workloads (shapes of the attention layers the source pages evaluate on,
which themselves need model weights and datasets not available here):
  single_head_decode  B=1, Hq=Hkv=1, D=64, Nk=256, one query; seed 0
  gqa_decode          B=8, Hq=32, Hkv=8, D=128, Nk=4096, one query each; K
                      has 4 outlier channels per kv-head scaled x10; seed 1
  long_decode         B=1, Hq=64, Hkv=8, D=128, Nk=131072, split-KV into
                      64-256 chunks (the bench takes 152: one per GB300 SM);
                      seed 2
  causal_prefill      B=2, Hq=32, Hkv=8, D=128, Nq=Nk=8192, causal; seed 3
  paged_decode        64 sequences, lengths uniform in [512, 32768], pages of
                      64 tokens in a randomly permuted pool, Hq=32, Hkv=8,
                      D=128; softmax scale 1/sqrt(D) and 1.0; seed 4
Q is fp16 ~ N(0, 1); K and V are fp32 ~ N(0, 1).
"""

from __future__ import annotations

import math

import numpy as np
import torch

WORKLOADS = {
    "single_head_decode": dict(kind="decode", B=1, Hq=1, Hkv=1, D=64, Nk=256, seed=0),
    "gqa_decode": dict(kind="decode", B=8, Hq=32, Hkv=8, D=128, Nk=4096, seed=1,
                       outliers=4, outlier_scale=10.0),
    "long_decode": dict(kind="decode", B=1, Hq=64, Hkv=8, D=128, Nk=131072, seed=2,
                        splits=(64, 128, 152, 256)),
    "causal_prefill": dict(kind="prefill", B=2, Hq=32, Hkv=8, D=128, Nq=8192, Nk=8192, seed=3),
    "paged_decode": dict(kind="paged", B=64, Hq=32, Hkv=8, D=128, len_lo=512, len_hi=32768,
                         page=64, seed=4, scales=(1.0 / math.sqrt(128), 1.0)),
}

_TAGS = {"q": 1, "k": 2, "v": 3, "outliers": 4, "lens": 5, "perm": 6}


def _generator(seed: int, tag: str, *idx: int) -> torch.Generator:
    s = int(seed) * 1_000_003 + _TAGS[tag] * 7919
    for i in idx:
        s = s * 131_071 + int(i) + 1
    g = torch.Generator()
    g.manual_seed(s % (2**63 - 1))
    return g


def queries(seed: int, *shape: int) -> torch.Tensor:
    """fp16 ~ N(0, 1) of the given shape ([B, Hq, D] or [B, Hq, Nq, D])."""
    return torch.randn(*shape, generator=_generator(seed, "q")).to(torch.float16)


def outlier_channels(seed: int, hkv: int, d: int, count: int) -> np.ndarray:
    """[hkv, count] channel indices drawn without replacement per kv-head."""
    out = np.zeros((hkv, count), dtype=np.int64)
    for h in range(hkv):
        out[h] = torch.randperm(d, generator=_generator(seed, "outliers", h))[:count].numpy()
    return out


def kv_slice(seed: int, which: str, b: int, kvh: int, n: int, d: int,
             outliers: np.ndarray | None = None, outlier_scale: float = 1.0) -> torch.Tensor:
    """fp32 [n, d] rows of K or V for (sequence b, kv-head kvh)."""
    x = torch.randn(n, d, generator=_generator(seed, which, b, kvh))
    if outliers is not None and which == "k":
        x[:, torch.as_tensor(outliers[kvh])] *= outlier_scale
    return x


def kv_block(seed: int, which: str, B: int, hkv: int, n: int, d: int,
             outliers: np.ndarray | None = None, outlier_scale: float = 1.0) -> torch.Tensor:
    """fp32 [B, hkv, n, d] built from independent slices."""
    out = torch.empty(B, hkv, n, d)
    for b in range(B):
        for h in range(hkv):
            out[b, h] = kv_slice(seed, which, b, h, n, d, outliers, outlier_scale)
    return out


def paged_layout(seed: int, B: int, len_lo: int, len_hi: int, page: int):
    """Random lengths (uniform integers in [len_lo, len_hi]) and a page table.

    Returns (lens int64 [B], page_table int32 [B, ceil(len_hi / page)] padded
    with -1, num_pages).  The pool holds exactly the pages needed, assigned
    through a random permutation.
    """
    g = _generator(seed, "lens")
    lens = torch.randint(len_lo, len_hi + 1, (B,), generator=g).numpy().astype(np.int64)
    need = (lens + page - 1) // page
    total = int(need.sum())
    perm = torch.randperm(total, generator=_generator(seed, "perm")).numpy()
    width = (len_hi + page - 1) // page
    table = -np.ones((B, width), dtype=np.int32)
    c = 0
    for b in range(B):
        table[b, : need[b]] = perm[c:c + need[b]]
        c += int(need[b])
    return lens, table, total
