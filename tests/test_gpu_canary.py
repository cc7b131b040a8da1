"""Out-of-bounds writes and tile edges, on the GPU.

compute-sanitizer is not available here, so every output of the public calls
is placed inside a larger buffer whose margins hold a fixed bit pattern; a
call must leave the margins untouched and write every element of its output.
The appended cache rows must be the only cache bytes a fused append changes.
Lengths sit on both sides of every tile edge of the kernels (32-token warp
slices, 64-token pages, 128-key prefill tiles, 256-row decode stages) and are
compared with the float64 oracle.
"""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, check_guards, guarded, require_gpu
from oracle import attention as att
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _oracle_decode(q, k, v, lens, scale):
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, LSE = att.attention_quantized(q.numpy()[:, :, None], pk, sk, pv, sv, scale, False, lens)
    return O[:, :, 0], LSE[:, :, 0]


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, lens, splits
    (3, 8, 2, 128, [1, 33, 257], 0),
    (3, 8, 2, 128, [1, 33, 257], 5),
    (2, 4, 4, 64, [65, 129], 0),
])
def test_decode_writes_only_its_outputs(case):
    qa = require_gpu()
    B, Hq, Hkv, D, lens, splits = case
    L = max(lens)
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(61, "k", B, Hkv, L, D), wl.kv_block(61, "v", B, Hkv, L, D)
    q = wl.queries(61, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, max(64, -(-L // 64) * 64), D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    ob, out = guarded((B, Hq, D), torch.float16)
    lb, lse = guarded((B, Hq), torch.float32)
    qa.decode(q.cuda(), cache, torch.tensor(lens, dtype=torch.int32).cuda(), L, scale, splits, out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    O, LSE = _oracle_decode(q, k, v, lens, scale)
    assert_close_attention(out, O)
    assert_close_lse(lse, LSE)
    assert qa.read_device_flags() == 0


def test_decode_append_changes_only_the_new_rows():
    qa = require_gpu()
    B, Hq, Hkv, D = 3, 16, 4, 128
    lens = [65, 1, 384]  # after the append: a page edge, a first token, a stage edge
    L, cap = max(lens), 448
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(62, "k", B, Hkv, L, D), wl.kv_block(62, "v", B, Hkv, L, D)
    q = wl.queries(62, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    for t in (cache.k_codes, cache.v_codes):  # rows past the lengths hold a pattern too
        for b, n in enumerate(lens):
            t[b, :, n:] = 0xA5
    for t in (cache.k_scales, cache.v_scales):
        for b, n in enumerate(lens):
            t[b, :, n:] = 0x3C00
    before = [t.clone() for t in (cache.k_codes, cache.v_codes, cache.k_scales, cache.v_scales)]
    idx = torch.tensor([n - 1 for n in lens])
    k_new = (k[torch.arange(B), :, idx] * 1.5).contiguous()  # differs from the rows it replaces
    v_new = (v[torch.arange(B), :, idx] * 1.5).contiguous()
    ob, out = guarded((B, Hq, D), torch.float16)
    lb, lse = guarded((B, Hq), torch.float32)
    qa.decode_append(q.cuda(), k_new.cuda(), v_new.cuda(), cache, torch.tensor(lens, dtype=torch.int32).cuda(),
                     L, scale, 0, out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    new_rows = np.zeros((B, Hkv, cap), dtype=bool)
    for b, n in enumerate(lens):
        new_rows[b, :, n - 1] = True
    mask = torch.from_numpy(new_rows).cuda()
    for name, old, now in zip(("k codes", "v codes", "k scales", "v scales"), before,
                              (cache.k_codes, cache.v_codes, cache.k_scales, cache.v_scales)):
        assert torch.equal(old[~mask], now[~mask]), f"{name}: a row other than the appended ones changed"
    pk_new, sk_new = codec.quantize_pack(k_new.numpy()[:, :, None])
    pv_new, sv_new = codec.quantize_pack(v_new.numpy()[:, :, None])
    for b, n in enumerate(lens):
        assert np.array_equal(cache.k_codes[b, :, n - 1].cpu().numpy(), pk_new[b, :, 0])
        assert np.array_equal(cache.v_codes[b, :, n - 1].cpu().numpy(), pv_new[b, :, 0])
        assert np.array_equal(cache.k_scales[b, :, n - 1].cpu().numpy().view(np.uint16), sk_new[b, :, 0].view(np.uint16))
        assert np.array_equal(cache.v_scales[b, :, n - 1].cpu().numpy().view(np.uint16), sv_new[b, :, 0].view(np.uint16))
    kh, vh = k.clone(), v.clone()
    for b, n in enumerate(lens):
        kh[b, :, n - 1], vh[b, :, n - 1] = k_new[b], v_new[b]
    O, LSE = _oracle_decode(q, kh, vh, lens, scale)
    assert_close_attention(out, O)
    assert_close_lse(lse, LSE)
    assert qa.read_device_flags() == 0


@pytest.mark.parametrize("nq,nk,causal", [(77, 300, True), (129, 129, True), (200, 257, False)])
def test_prefill_writes_only_its_outputs(nq, nk, causal):
    qa = require_gpu()
    B, Hq, Hkv, D = 2, 4, 2, 128
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(63, "k", B, Hkv, nk, D), wl.kv_block(63, "v", B, Hkv, nk, D)
    q = wl.queries(63, B, Hq, nq, D)
    cache = qa.KvCache.contiguous(B, Hkv, -(-nk // 64) * 64, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    ob, out = guarded((B, Hq, nq, D), torch.float16)
    lb, lse = guarded((B, Hq, nq), torch.float32)
    qa.prefill(q.cuda(), cache, nk, scale, causal, out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, LSE = att.attention_quantized(q.numpy(), pk, sk, pv, sv, scale, causal)
    assert_close_attention(out, O)
    assert_close_lse(lse, LSE)
    assert qa.read_device_flags() == 0


def test_combine_writes_only_its_outputs():
    qa = require_gpu()
    S, R, D = 5, 37, 128
    g = torch.Generator().manual_seed(64)
    po = torch.randn(S, R, D, generator=g)
    pl = torch.randn(S, R, generator=g) * 3
    pl[1, 3] = -math.inf  # a split that saw no key
    pl[:, 7] = -math.inf  # a row no split saw: O = 0, lse = -inf
    ob, out = guarded((R, D), torch.float16)
    lb, lse = guarded((R,), torch.float32)
    qa.combine(po.cuda(), pl.cuda(), out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    O, LSE = att.combine(po.numpy().astype(np.float64), pl.numpy().astype(np.float64))
    assert_close_attention(out, O, max_abs=1e-3, mean_abs=2e-4)
    assert_close_lse(lse, LSE, tol=1e-5)


EDGE_LENS = [1, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]


@pytest.mark.parametrize("splits", [0, 3])
def test_decode_tile_edge_lengths(splits):
    qa = require_gpu()
    B, Hq, Hkv, D = len(EDGE_LENS), 8, 2, 128
    L = max(EDGE_LENS)
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(65, "k", B, Hkv, L, D), wl.kv_block(65, "v", B, Hkv, L, D)
    q = wl.queries(65, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, 320, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    out, lse = qa.decode(q.cuda(), cache, torch.tensor(EDGE_LENS, dtype=torch.int32).cuda(), L, scale, splits,
                         return_lse=True)
    O, LSE = _oracle_decode(q, k, v, EDGE_LENS, scale)
    assert_close_attention(out, O)
    assert_close_lse(lse, LSE)
    assert qa.read_device_flags() == 0


@pytest.mark.parametrize("n", [1, 63, 64, 65, 127, 128, 129])
def test_prefill_tile_edge_lengths(n):
    qa = require_gpu()
    B, Hq, Hkv, D = 1, 2, 1, 128
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(66, "k", B, Hkv, n, D), wl.kv_block(66, "v", B, Hkv, n, D)
    q = wl.queries(66, B, Hq, n, D)
    cache = qa.KvCache.contiguous(B, Hkv, max(64, -(-n // 64) * 64), D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    out, lse = qa.prefill(q.cuda(), cache, n, scale, True, return_lse=True)
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, LSE = att.attention_quantized(q.numpy(), pk, sk, pv, sv, scale, True)
    assert_close_attention(out, O)
    assert_close_lse(lse, LSE)
    assert qa.read_device_flags() == 0
