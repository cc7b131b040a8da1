"""GPU parity of qattn_decode (split-KV, contiguous and paged) against the oracle."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, require_gpu
from oracle import attention as att
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _run_contiguous(seed, B, Hq, Hkv, D, lens, splits, scale, outliers=False):
    qa = require_gpu()
    L = max(max(lens), 1)
    cap = max(64, -(-L // 64) * 64)
    oc = wl.outlier_channels(seed, Hkv, D, 4) if outliers else None
    k = wl.kv_block(seed, "k", B, Hkv, L, D, oc, 10.0)
    v = wl.kv_block(seed, "v", B, Hkv, L, D)
    q = wl.queries(seed, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    sl = torch.tensor(lens, dtype=torch.int32)
    out, lse = qa.decode(q.cuda(), cache, sl.cuda(), L, scale, splits, return_lse=True)
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, LSE = att.attention_quantized(q.numpy()[:, :, None], pk, sk, pv, sv, scale, False, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, LSE[:, :, 0])
    assert qa.read_device_flags() == 0


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, lens, splits, scale
    (1, 1, 1, 64, [256], 0, 1 / 8),                      # single-head decode shape
    (3, 8, 2, 128, [1, 100, 777], 1, 1 / math.sqrt(128)),
    (3, 8, 2, 128, [1, 100, 777], 0, 1 / math.sqrt(128)),
    (3, 8, 2, 128, [0, 64, 777], 7, 1 / math.sqrt(128)),  # empty sequence, ragged tails
    (2, 16, 2, 128, [1000, 513], 5, 1.0),                 # G = 8, softmax scale 1.0
    (2, 4, 4, 64, [129, 65], 3, 1 / 8),                   # G = 1, D = 64
    (2, 12, 4, 128, [300, 200], 2, 0.1),                  # G = 3
    (1, 64, 8, 128, [4096], 64, 1 / math.sqrt(128)),      # long-context shape, many splits
    (1, 8, 1, 128, [40000], 64, 1.0),                     # one segment over 64 splits: two merge batches
    # long ranges (>= 12 stages of 384 tokens per range): the 12-warp layout
    (3, 16, 4, 128, [20000, 0, 9001], 4, 1 / math.sqrt(128)),
    (2, 8, 2, 64, [16000, 15999], 2, 1 / 8),
    (1, 32, 4, 128, [40000], 3, 1.0),                      # G = 8, softmax scale 1.0
])
def test_decode_contiguous(case):
    B, Hq, Hkv, D, lens, splits, scale = case
    _run_contiguous(17, B, Hq, Hkv, D, lens, splits, scale)


def test_decode_outlier_channels():
    _run_contiguous(1, 2, 32, 8, 128, [4096, 1000], 0, 1 / math.sqrt(128), outliers=True)


def _run_paged(seed, B, Hq, Hkv, D, lo, hi, splits, scale):
    qa = require_gpu()
    lens, table, P = wl.paged_layout(seed, B, lo, hi, 64)
    cache = qa.KvCache.paged(P, Hkv, D, torch.from_numpy(table))
    O = np.zeros((B, Hq, D))
    LSE = np.zeros((B, Hq))
    q = wl.queries(seed, B, Hq, D)
    for b, n in enumerate(lens):
        n = int(n)
        k = torch.stack([wl.kv_slice(seed, "k", b, h, n, D) for h in range(Hkv)])[None]
        v = torch.stack([wl.kv_slice(seed, "v", b, h, n, D) for h in range(Hkv)])[None]
        sub = qa.KvCache(cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales, D, Hkv,
                         page_table=cache.page_table[b:b + 1], num_pages=P)
        qa.quantize_kv(k.cuda(), v.cuda(), sub)
        pk, sk = codec.quantize_pack(k.numpy())
        pv, sv = codec.quantize_pack(v.numpy())
        o, l = att.attention_quantized(q.numpy()[b:b + 1, :, None], pk, sk, pv, sv, scale)
        O[b], LSE[b] = o[0, :, 0], l[0, :, 0]
    out, lse = qa.decode(q.cuda(), cache, torch.from_numpy(lens).cuda(), int(hi), scale, splits,
                         return_lse=True)
    assert_close_attention(out, O)
    assert_close_lse(lse, LSE)
    assert qa.read_device_flags() == 0


@pytest.mark.parametrize("splits", [0, 1, 6])
@pytest.mark.parametrize("scale", [1 / math.sqrt(128), 1.0])
def test_decode_paged(splits, scale):
    _run_paged(23, 5, 32, 8, 128, 1, 700, splits, scale)


def test_decode_paged_d64_g1():
    _run_paged(29, 4, 2, 2, 64, 60, 300, 0, 1 / 8)


def test_split_count_does_not_change_the_result():
    qa = require_gpu()
    B, Hq, Hkv, D, L = 2, 8, 2, 128, 1500
    k = wl.kv_block(3, "k", B, Hkv, L, D)
    v = wl.kv_block(3, "v", B, Hkv, L, D)
    q = wl.queries(3, B, Hq, D).cuda()
    cache = qa.KvCache.contiguous(B, Hkv, L, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    sl = torch.tensor([L, 999], dtype=torch.int32).cuda()
    outs = [qa.decode(q, cache, sl, L, 0.1, s, return_lse=True) for s in (1, 2, 5, 24)]
    for o, l in outs[1:]:
        _close_to_unsplit(o, l, *outs[0], cache)


def _close_to_unsplit(o, l, o1, l1, cache):
    """The split-KV merge against the unsplit result of the same kernel.  lse
    within 1e-5 relative: the log-sum-exp combine and the fp32 sums of p are
    exact up to fp32 rounding.  O: its numerator sums the fp16-rounded P'
    (relative error 2^-11 each) while the normaliser sums p in fp32, and the
    split cuts the keys into other chunks, so O moves by up to 2 * 2^-11 of
    the largest |v^| (7 * the largest V scale), plus one fp16 ulp of O."""
    o, o1 = o.float(), o1.float()
    assert ((l - l1).abs() <= 1e-5 * l1.abs() + 1e-6).all(), (l - l1).abs().max().item()
    vmax = 7.0 * cache.v_scales.float().abs().max().item()
    tol = 2 * 2.0**-11 * vmax + o1.abs() * 2.0**-10
    assert ((o - o1).abs() <= tol).all(), (o - o1).abs().max().item()


def test_long_context_splits_match_one_range():
    """The long-context shape (B = 1, Hq = 64, Hkv = 8, D = 128, 131072 tokens):
    the automatic split (one range per SM, merged) against a single range."""
    qa = require_gpu()
    B, Hq, Hkv, D, N = 1, 64, 8, 128, 131072
    g = torch.Generator(device="cuda")
    g.manual_seed(97)
    cache = qa.KvCache.contiguous(B, Hkv, N, D)
    qa.quantize_kv(torch.randn(B, Hkv, N, D, device="cuda", generator=g),
                   torch.randn(B, Hkv, N, D, device="cuda", generator=g), cache)
    q = torch.randn(B, Hq, D, device="cuda", generator=g).half()
    sl = torch.full((B,), N, dtype=torch.int32, device="cuda")
    o1, l1 = qa.decode(q, cache, sl, N, 1 / math.sqrt(D), 1, return_lse=True)
    o, l = qa.decode(q, cache, sl, N, 1 / math.sqrt(D), 0, return_lse=True)
    _close_to_unsplit(o, l, o1, l1, cache)
    assert qa.read_device_flags() == 0
