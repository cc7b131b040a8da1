"""GPU parity of the FlashQ-style decode buffer (qattn_flashq_*) against the
step-by-step oracle (oracle/flashq.py): TurboAttention §3.3.

Every case replays decode steps: append one K/V row per (sequence, kv-head)
to the buffer, decode over the cached rows, merge the buffered rows in; at
64 buffered rows the buffer is flushed into the INT4 cache.  Buffered int8
codes, universal scales, ranges and flushed INT4 rows are checked bit for
bit every step; O and lse against the float64 oracle.
"""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, check_guards, guarded, require_gpu
from oracle import codec
from oracle import flashq as fq
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


def _replay(seed, B, Hq, Hkv, D, L0, steps, paged=False, dt=torch.float32, outlier_step=None):
    qa = require_gpu()
    G = Hq // Hkv
    scale = 1 / math.sqrt(D)
    cap = -(-(L0 + 64 * (steps // 64 + 1)) // 64) * 64
    hk = wl.kv_block(seed, "k", B, Hkv, L0, D)
    hv = wl.kv_block(seed, "v", B, Hkv, L0, D)
    if paged:
        pages = cap // 64
        table = torch.arange(B * pages, dtype=torch.int32).reshape(B, pages)
        table = table[:, torch.randperm(pages, generator=torch.Generator().manual_seed(seed))].contiguous()
        cache = qa.KvCache.paged(B * pages, Hkv, D, table)
    else:
        cache = qa.KvCache.contiguous(B, Hkv, cap, D)
    if L0:
        qa.quantize_kv(hk.cuda(), hv.cuda(), cache)
    heads = [[(fq.BufferedHead(hk[b, h].numpy()), fq.BufferedHead(hv[b, h].numpy())) for h in range(Hkv)]
             for b in range(B)]
    buf = qa.FlashqBuffer.create(B, Hkv, D)
    cache_len = L0
    qa.flashq_init(buf, cache, torch.full((B,), cache_len, dtype=torch.int32))
    torch.cuda.synchronize()
    for b in range(B):
        for h in range(Hkv):
            assert buf.k_range[b, h].item() == float(heads[b][h][0].r)
            assert _bits(buf.v_scale[b, h]) == np.float16(heads[b][h][1].u).view(np.uint16)
    nk = wl.kv_block(seed + 1, "k", B, Hkv, steps, D)
    nv = wl.kv_block(seed + 1, "v", B, Hkv, steps, D)
    if outlier_step is not None:
        nk[:, :, outlier_step] *= 20.0  # past the universal range: clamped
    for s in range(steps):
        kn, vn = nk[:, :, s].contiguous(), nv[:, :, s].contiguous()
        qa.flashq_append(kn.to(dt).cuda(), vn.to(dt).cuda(), buf)
        slot = s % fq.NB
        for b in range(B):
            for h in range(Hkv):
                ck = heads[b][h][0].append(kn[b, h].to(dt).float().numpy())
                cv = heads[b][h][1].append(vn[b, h].to(dt).float().numpy())
                assert np.array_equal(buf.k_codes[b, h, slot].cpu().numpy(), ck), (s, b, h)
                assert np.array_equal(buf.v_codes[b, h, slot].cpu().numpy(), cv), (s, b, h)
        q = wl.queries(seed + 100 + s, B, Hq, D)
        ob, out = guarded((B, Hq, D), torch.float16)
        lb, lse = guarded((B, Hq), torch.float32)
        qa.decode(q.cuda(), cache, torch.full((B,), cache_len, dtype=torch.int32).cuda(), cache_len + 64, scale, 0,
                  out=out, lse=lse)
        qa.flashq_attend(q.cuda(), buf, scale, out, lse)
        torch.cuda.synchronize()
        check_guards(ob, "out")
        check_guards(lb, "lse")
        O = np.zeros((B, Hq, D))
        LSE = np.zeros((B, Hq))
        for b in range(B):
            for h in range(Hkv):
                o, l = fq.attention_buffered(q.numpy()[b, h * G:(h + 1) * G], heads[b][h][0], heads[b][h][1], scale)
                O[b, h * G:(h + 1) * G], LSE[b, h * G:(h + 1) * G] = o, l
        assert_close_attention(out, O)
        assert_close_lse(lse, LSE)
        if slot == fq.NB - 1:  # the buffer is full: into the cache
            qa.flashq_flush(buf, cache, torch.full((B,), cache_len, dtype=torch.int32))
            torch.cuda.synchronize()
            for b in range(B):
                for h in range(Hkv):
                    for t, hd in enumerate(heads[b][h]):
                        p, sc = hd.flush()
                        codes = cache.v_codes if t else cache.k_codes
                        scales = cache.v_scales if t else cache.k_scales
                        for i in range(fq.NB):
                            pos = cache_len + i
                            if paged:
                                page = int(cache.page_table[b, pos // 64])
                                got_c, got_s = codes[page, h, pos % 64], scales[page, h, pos % 64]
                            else:
                                got_c, got_s = codes[b, h, pos], scales[b, h, pos]
                            assert np.array_equal(got_c.cpu().numpy(), p[i]), (b, h, t, i)
                            assert _bits(got_s) == sc[i].view(np.uint16)
                        rng_t = buf.v_range if t else buf.k_range
                        sc_t = buf.v_scale if t else buf.k_scale
                        assert rng_t[b, h].item() == float(hd.r)
                        assert _bits(sc_t[b, h]) == np.float16(hd.u).view(np.uint16)
            assert buf.count.cpu().tolist() == [0] * B
            cache_len += fq.NB
    assert qa.read_device_flags() == 0


def test_flashq_steps_with_history():
    _replay(41, 2, 8, 2, 128, 300, 70, outlier_step=5)


def test_flashq_empty_history_fp16_rows():
    _replay(43, 2, 4, 1, 128, 0, 66, dt=torch.float16)


def test_flashq_paged_d64():
    _replay(47, 2, 8, 4, 64, 129, 65, paged=True)


def test_flashq_full_buffer_is_flagged():
    qa = require_gpu()
    buf = qa.FlashqBuffer.create(1, 1, 64)
    cache = qa.KvCache.contiguous(1, 1, 64, 64)
    qa.flashq_init(buf, cache, torch.zeros(1, dtype=torch.int32))
    row = torch.ones(1, 1, 64).cuda()
    for _ in range(fq.NB):
        qa.flashq_append(row, row, buf)
    qa.read_device_flags(clear=True)
    qa.flashq_append(row, row, buf)
    assert qa.read_device_flags(clear=True) & qa.FLAG_BUFFER_FULL
    assert buf.count.item() == fq.NB


def test_flashq_group_of_eight():
    """G = 8, as in the long-context shape the bench times."""
    _replay(53, 1, 16, 2, 128, 200, 66)
