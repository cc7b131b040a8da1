"""GPU parity of qattn_decode_append: one launch that quantizes each
sequence's new K/V row into the cache and attends over it.

Each case runs the fused step and, on a second copy of the cache, the two-call
form (qattn_quantize_kv of the new row, then qattn_decode).  The caches must
match bit for bit and so must O and lse (the same decode path reads the same
bytes); the float64 oracle then checks the new row's codes and scales and O
against its own quantization of the whole K/V history.
"""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, require_gpu
from oracle import attention as att
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _clone(qa, cache):
    return qa.KvCache(cache.k_codes.clone(), cache.k_scales.clone(), cache.v_codes.clone(), cache.v_scales.clone(),
                      cache.head_dim, cache.num_kv_heads, capacity=cache.capacity,
                      page_table=cache.page_table, num_pages=cache.num_pages)


def _same_cache(a, b):
    for x, y in ((a.k_codes, b.k_codes), (a.v_codes, b.v_codes), (a.k_scales, b.k_scales), (a.v_scales, b.v_scales)):
        assert torch.equal(x, y)


def _history(seed, B, Hkv, L, D):
    """K/V of L positions per (sequence, kv-head); the last used one is the new row."""
    return wl.kv_block(seed, "k", B, Hkv, L, D), wl.kv_block(seed, "v", B, Hkv, L, D)


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, lens (after the append), splits, new-row dtype
    (3, 8, 2, 128, [1, 100, 777], 0, torch.float32),
    (3, 8, 2, 128, [64, 65, 256], 5, torch.float16),      # new row first / last in a stage
    (2, 4, 4, 64, [0, 129], 3, torch.float32),            # empty sequence: nothing appended
    (1, 64, 8, 128, [4096], 152, torch.float32),          # long-context shape, many splits
    (2, 16, 2, 128, [20000, 9001], 4, torch.float16),     # 12-warp layout
])
def test_decode_append_contiguous(case):
    qa = require_gpu()
    B, Hq, Hkv, D, lens, splits, dt = case
    seed = 23
    L = max(max(lens), 1)
    cap = max(64, -(-L // 64) * 64)
    k, v = _history(seed, B, Hkv, L, D)
    q = wl.queries(seed, B, Hq, D)
    scale = 1 / math.sqrt(D)
    a = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), a)  # the history; the new rows are written again below
    for b, n in enumerate(lens):           # ... so clear them first: they must come from the append
        if n > 0:
            a.k_codes[b, :, n - 1] = 0
            a.v_codes[b, :, n - 1] = 0
            a.k_scales[b, :, n - 1] = 0
            a.v_scales[b, :, n - 1] = 0
    c = _clone(qa, a)
    idx = torch.tensor([max(n - 1, 0) for n in lens])
    k_new = k[torch.arange(B), :, idx].to(dt).contiguous()  # [B, Hkv, D]
    v_new = v[torch.arange(B), :, idx].to(dt).contiguous()
    sl = torch.tensor(lens, dtype=torch.int32).cuda()
    out, lse = qa.decode_append(q.cuda(), k_new.cuda(), v_new.cuda(), a, sl, L, scale, splits, return_lse=True)
    # the two-call form
    qa.quantize_kv(k_new[:, :, None].cuda(), v_new[:, :, None].cuda(), c,
                   torch.tensor([max(n - 1, 0) if n > 0 else cap for n in lens], dtype=torch.int32).cuda())
    out2, lse2 = qa.decode(q.cuda(), c, sl, L, scale, splits, return_lse=True)
    torch.cuda.synchronize()
    _same_cache(a, c)
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)
    # the oracle on the whole history (new rows as the dtype they were given)
    kh, vh = k.clone(), v.clone()
    for b, n in enumerate(lens):
        if n > 0:
            kh[b, :, n - 1] = k_new[b].float()
            vh[b, :, n - 1] = v_new[b].float()
    pk, sk = codec.quantize_pack(kh.numpy())
    pv, sv = codec.quantize_pack(vh.numpy())
    for b, n in enumerate(lens):
        if n > 0:
            assert np.array_equal(a.k_codes[b, :, n - 1].cpu().numpy(), pk[b, :, n - 1])
            assert np.array_equal(a.v_codes[b, :, n - 1].cpu().numpy(), pv[b, :, n - 1])
            assert np.array_equal(a.k_scales[b, :, n - 1].cpu().numpy().view(np.uint16), sk[b, :, n - 1].view(np.uint16))
            assert np.array_equal(a.v_scales[b, :, n - 1].cpu().numpy().view(np.uint16), sv[b, :, n - 1].view(np.uint16))
    O, LSE = att.attention_quantized(q.numpy()[:, :, None], pk, sk, pv, sv, scale, False, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, LSE[:, :, 0])
    assert qa.read_device_flags() == 0


def test_decode_append_paged():
    qa = require_gpu()
    seed, B, Hq, Hkv, D, splits = 29, 5, 32, 8, 128, 0
    lens, table, P = wl.paged_layout(seed, B, 100, 700, 64)
    lens[0], lens[1] = 64, 65  # the new row last in a page / first in a new page (pages exist for >= 100)
    a = qa.KvCache.paged(P, Hkv, D, torch.from_numpy(table))
    q = wl.queries(seed, B, Hq, D)
    scale = 1 / math.sqrt(D)
    L = int(lens.max())
    k, v = _history(seed, B, Hkv, L, D)
    for b, n in enumerate(lens):  # the history without the new row
        n = int(n)
        if n > 1:
            sub = qa.KvCache(a.k_codes, a.k_scales, a.v_codes, a.v_scales, D, Hkv,
                             page_table=a.page_table[b:b + 1], num_pages=P)
            qa.quantize_kv(k[b:b + 1, :, :n - 1].contiguous().cuda(), v[b:b + 1, :, :n - 1].contiguous().cuda(), sub)
    idx = torch.tensor([int(n) - 1 for n in lens])
    k_new = k[torch.arange(B), :, idx].contiguous()
    v_new = v[torch.arange(B), :, idx].contiguous()
    sl = torch.from_numpy(lens).cuda()
    out, lse = qa.decode_append(q.cuda(), k_new.cuda(), v_new.cuda(), a, sl, L, scale, splits, return_lse=True)
    torch.cuda.synchronize()
    O = np.zeros((B, Hq, D))
    LSE = np.zeros((B, Hq))
    for b, n in enumerate(lens):
        n = int(n)
        pk, sk = codec.quantize_pack(k[b:b + 1, :, :n].numpy())
        pv, sv = codec.quantize_pack(v[b:b + 1, :, :n].numpy())
        o, l = att.attention_quantized(q.numpy()[b:b + 1, :, None], pk, sk, pv, sv, scale)
        O[b], LSE[b] = o[0, :, 0], l[0, :, 0]
        page = int(table[b, (n - 1) // 64])
        got_k = a.k_codes[page, :, (n - 1) % 64].cpu().numpy()
        assert np.array_equal(got_k, pk[0, :, n - 1])
        got_sv = a.v_scales[page, :, (n - 1) % 64].cpu().numpy().view(np.uint16)
        assert np.array_equal(got_sv, sv[0, :, n - 1].view(np.uint16))
    assert_close_attention(out, O)
    assert_close_lse(lse, LSE)
    assert qa.read_device_flags() == 0


def test_decode_append_beyond_capacity_is_flagged():
    """A new row past the cache is not written; the length is clamped and flagged."""
    qa = require_gpu()
    B, Hq, Hkv, D, cap = 1, 4, 1, 64, 128
    k, v = _history(31, B, Hkv, cap, D)
    a = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), a)
    before = _clone(qa, a)
    q = wl.queries(31, B, Hq, D)
    new = torch.ones(B, Hkv, D)
    qa.read_device_flags(clear=True)
    out = qa.decode_append(q.cuda(), new.cuda(), new.cuda(), a, torch.tensor([cap + 1], dtype=torch.int32).cuda(),
                           cap + 1, 1 / 8)
    torch.cuda.synchronize()
    _same_cache(a, before)
    assert qa.read_device_flags(clear=True) & qa.FLAG_BAD_PAGE
    ref = qa.decode(q.cuda(), before, torch.tensor([cap], dtype=torch.int32).cuda(), cap, 1 / 8)
    assert torch.equal(out, ref)
