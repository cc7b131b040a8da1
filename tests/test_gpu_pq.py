"""GPU parity of progressive INT8 -> INT4 storage (TurboAttention §3.1):
qattn_pq_quantize bit for bit against oracle/progressive (codes, s2, z2, s1,
the record's zero padding), and qattn_decode_pq within the attention
tolerance of float64 attention over the oracle's dequantized blocks."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, check_guards, guarded, require_gpu
from oracle import progressive as pq
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _records(params, D):
    p = params.cpu().numpy()
    s2 = p[..., :D]
    z2 = p[..., D:2 * D].view(np.int8)
    s1 = p[..., 2 * D:2 * D + 2].copy().view(np.float16)[..., 0]
    pad = p[..., 2 * D + 2:]
    return s2, z2, s1, pad


@pytest.mark.parametrize("case", [
    # B, Hkv, n, D, dtype, start_blocks
    (2, 3, 192, 128, torch.float32, None),
    (1, 2, 128, 64, torch.float16, [2]),
    (3, 1, 64, 128, torch.float32, [0, 5, 1]),
])
def test_pq_quantize_matches_oracle_bits(case):
    qa = require_gpu()
    B, Hkv, n, D, dt, starts = case
    k = wl.kv_block(71, "k", B, Hkv, n, D)
    v = wl.kv_block(71, "v", B, Hkv, n, D)
    k[0, 0, :, 3] *= 10.0                      # an outlier channel
    if B > 1:
        k[1, 0, :64] = 0.0                     # an all-zero block: s1 = 0, codes 0
    k, v = k.to(dt), v.to(dt)
    cap = 512
    cache = qa.PqCache.contiguous(B, Hkv, cap, D)
    sb = None if starts is None else torch.tensor(starts, dtype=torch.int32)
    qa.pq_quantize(k.cuda(), v.cuda(), cache, None if sb is None else sb.cuda())
    torch.cuda.synchronize()
    for x, codes, params in ((k, cache.k_codes, cache.k_params), (v, cache.v_codes, cache.v_params)):
        wp, ws1, ws2, wz2 = pq.quantize_blocks(x.float().numpy())
        s2, z2, s1, pad = _records(params, D)
        for b in range(B):
            b0 = 0 if starts is None else starts[b]
            nb = n // 64
            got_codes = codes[b, :, b0 * 64:(b0 + nb) * 64].cpu().numpy()
            assert np.array_equal(got_codes, wp[b])
            assert np.array_equal(s2[b, :, b0:b0 + nb], ws2[b])
            assert np.array_equal(z2[b, :, b0:b0 + nb], wz2[b])
            assert np.array_equal(s1[b, :, b0:b0 + nb].view(np.uint16), ws1[b].view(np.uint16))
            assert not pad[b, :, b0:b0 + nb].any()
    assert qa.read_device_flags() == 0


def test_pq_quantize_flags_blocks_past_the_cache():
    qa = require_gpu()
    cache = qa.PqCache.contiguous(1, 1, 128, 64)
    x = torch.randn(1, 1, 128, 64)
    qa.pq_quantize(x.cuda(), x.cuda(), cache, torch.tensor([1], dtype=torch.int32).cuda())   # blocks 1, 2 of 2
    assert qa.read_device_flags() == qa.FLAG_BAD_PAGE
    assert cache.k_codes[0, 0, 64:].any()                     # block 1 was written


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, lens, splits, scale
    (3, 16, 4, 128, [1024, 512, 64], 0, 1 / math.sqrt(128)),
    (3, 16, 4, 128, [1024, 512, 64], 1, 1 / math.sqrt(128)),
    (3, 16, 4, 128, [1024, 700, 0], 5, 1.0),          # a length inside a block; an empty sequence
    (2, 4, 4, 64, [320, 128], 3, 0.125),              # G = 1
    (1, 64, 8, 128, [4096], 0, 1 / math.sqrt(128)),   # G = 8, many ranges
])
def test_decode_pq_matches_oracle(case):
    qa = require_gpu()
    B, Hq, Hkv, D, lens, splits, scale = case
    cap = max(64, -(-max(lens) // 64) * 64)
    k = wl.kv_block(72, "k", B, Hkv, cap, D)
    v = wl.kv_block(72, "v", B, Hkv, cap, D)
    cache = qa.PqCache.contiguous(B, Hkv, cap, D)
    qa.pq_quantize(k.cuda(), v.cuda(), cache)
    q = wl.queries(72, B, Hq, D)
    ob, out = guarded((B, Hq, D), torch.float16)
    lb, lse = guarded((B, Hq), torch.float32)
    qa.decode_pq(q.cuda(), cache, torch.tensor(lens, dtype=torch.int32), max(lens), scale, splits, out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    O, L = pq.attention_pq(q.numpy()[:, :, None], pq.quantize_blocks(k.numpy()), pq.quantize_blocks(v.numpy()),
                           scale, False, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, L[:, :, 0])
    assert qa.read_device_flags() == 0


def test_flashq_flush_into_progressive_blocks():
    """A full decode buffer -> one block: stage 2 on the buffer's own int8
    codes with s1 = its universal scale, bit for bit; the buffer empties, R
    and u stay; the flushed block then decodes like the oracle's."""
    qa = require_gpu()
    from oracle import flashq as fq
    B, Hq, Hkv, D, L0 = 2, 8, 2, 128, 192
    hk = wl.kv_block(73, "k", B, Hkv, L0, D)
    hv = wl.kv_block(73, "v", B, Hkv, L0, D)
    cache4 = qa.KvCache.contiguous(B, Hkv, L0 + 64, D)
    qa.quantize_kv(hk.cuda(), hv.cuda(), cache4)
    heads = [[(fq.BufferedHead(hk[b, h].numpy()), fq.BufferedHead(hv[b, h].numpy())) for h in range(Hkv)]
             for b in range(B)]
    buf = qa.FlashqBuffer.create(B, Hkv, D)
    qa.flashq_init(buf, cache4, torch.full((B,), L0, dtype=torch.int32))
    nk = wl.kv_block(74, "k", B, Hkv, 64, D)
    nv = wl.kv_block(74, "v", B, Hkv, 64, D)
    nk[:, :, 17] *= 20.0                                       # outliers: clamped into the universal range
    for s in range(64):
        qa.flashq_append(nk[:, :, s].contiguous().cuda(), nv[:, :, s].contiguous().cuda(), buf)
        for b in range(B):
            for h in range(Hkv):
                heads[b][h][0].append(nk[b, h, s].numpy())
                heads[b][h][1].append(nv[b, h, s].numpy())
    ranges = (buf.k_range.clone(), buf.v_range.clone(), buf.k_scale.clone(), buf.v_scale.clone())
    cap = 256
    pqc = qa.PqCache.contiguous(B, Hkv, cap, D)
    pos = torch.tensor([64, 128], dtype=torch.int32)           # block positions 1 and 2
    qa.flashq_flush_pq(buf, pqc, pos.cuda())
    torch.cuda.synchronize()
    assert buf.count.cpu().tolist() == [0, 0]
    for a, b_ in zip(ranges, (buf.k_range, buf.v_range, buf.k_scale, buf.v_scale)):
        assert torch.equal(a, b_)
    stores = []
    for t, (codes, params) in enumerate(((pqc.k_codes, pqc.k_params), (pqc.v_codes, pqc.v_params))):
        s2, z2, s1, pad = _records(params, D)
        per_b = []
        for b in range(B):
            blk = int(pos[b]) // 64
            per_h = []
            for h in range(Hkv):
                head = heads[b][h][t]
                wp, ws1, ws2, wz2 = pq.compress_int8_block(np.stack(head.codes), head.u)
                assert np.array_equal(codes[b, h, blk * 64:(blk + 1) * 64].cpu().numpy(), wp)
                assert np.array_equal(s2[b, h, blk], ws2) and np.array_equal(z2[b, h, blk], wz2)
                assert s1[b, h, blk].view(np.uint16) == np.float16(ws1).view(np.uint16)
                assert not pad[b, h, blk].any()
                per_h.append((wp, ws1, ws2, wz2))
            per_b.append(per_h)
        stores.append(per_b)
    # decode over each sequence's keys up to the end of its flushed block: the
    # blocks before it were never written (zero records), so their values are 0
    q = wl.queries(75, B, Hq, D)
    scale = 1 / math.sqrt(D)
    lens = (pos + 64).tolist()
    out = qa.decode_pq(q.cuda(), pqc, torch.tensor(lens, dtype=torch.int32), max(lens), scale, 0)
    O = np.zeros((B, Hq, D))
    for b in range(B):
        blk = int(pos[b]) // 64

        def values(t):  # [1, Hkv, lens[b], D]: zeros, then the flushed block
            rows = []
            for h in range(Hkv):
                wp, ws1, ws2, wz2 = stores[t][b][h]
                blkv = pq.dequantize_blocks(wp, np.array([ws1]), ws2[None], wz2[None])
                rows.append(np.concatenate([np.zeros((blk * 64, D)), blkv]))
            return np.stack(rows)[None]
        o, _ = pq.att.attention(q.numpy()[b:b + 1, :, None], values(0), values(1), scale)
        O[b] = o[0, :, 0]
    assert_close_attention(out, O)
    assert qa.read_device_flags() == 0
