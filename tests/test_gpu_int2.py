"""GPU parity of the INT2 cache (TurboAttention, arXiv 2412.08585, §3.2's
2-bit heads in this library's per-row symmetric layout: sixteen 2-bit values
per 32-bit word) against oracle/codec2: the append's words and scales bit for
bit, and split-KV decode over the INT2 rows against float64 attention over
their dequantized values."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, check_guards, guarded, require_gpu
from oracle import attention as att
from oracle import codec2 as c2
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _words(t):
    """uint8 [..., 32] -> little-endian uint32 [..., 8]."""
    return t.cpu().numpy().view(np.uint32)


def _fill(qa, seed, B, Hkv, L, D=128, dt=torch.float32):
    cap = max(64, -(-L // 64) * 64)
    k = wl.kv_block(seed, "k", B, Hkv, L, D)
    v = wl.kv_block(seed, "v", B, Hkv, L, D)
    cache = qa.KvCache.contiguous(B, Hkv, cap, D, code_bits=2)
    qa.quantize_kv(k.to(dt).cuda(), v.to(dt).cuda(), cache)
    torch.cuda.synchronize()
    return cache, k.to(dt).float(), v.to(dt).float()


@pytest.mark.parametrize("dt", [torch.float32, torch.float16])
def test_int2_append_is_bit_exact(dt):
    qa = require_gpu()
    cache, k, v = _fill(qa, 71, 2, 3, 200, dt=dt)
    for x, codes, scales in ((k, cache.k_codes, cache.k_scales), (v, cache.v_codes, cache.v_scales)):
        w, s = c2.quantize_pack2(x.numpy())
        assert np.array_equal(_words(codes[:, :, :200]), w)
        assert np.array_equal(scales[:, :, :200].cpu().numpy().view(np.uint16), s.view(np.uint16))


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, lens, splits, scale
    (3, 8, 2, [1, 100, 777], 0, 1 / math.sqrt(128)),
    (3, 8, 2, [0, 64, 777], 5, 1 / math.sqrt(128)),      # empty sequence, ragged tails
    (2, 16, 2, [1000, 513], 3, 1.0),                     # G = 8, softmax scale 1.0
    (2, 4, 4, [129, 300], 2, 1 / math.sqrt(128)),        # G = 1
    (2, 12, 4, [300, 200], 2, 0.1),                      # G = 3
    (1, 64, 8, [4096], 64, 1 / math.sqrt(128)),          # long-context shape, many splits
    (2, 16, 2, [20000, 9001], 4, 1 / math.sqrt(128)),    # long ranges, few splits
])
def test_int2_decode(case):
    qa = require_gpu()
    B, Hq, Hkv, lens, splits, scale = case
    L = max(max(lens), 1)
    cache, k, v = _fill(qa, 73, B, Hkv, L)
    q = wl.queries(73, B, Hq, 128)
    ob, out = guarded((B, Hq, 128), torch.float16)
    lb, lse = guarded((B, Hq), torch.float32)
    qa.decode(q.cuda(), cache, torch.tensor(lens, dtype=torch.int32).cuda(), L, scale, splits, out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    wk, sk = c2.quantize_pack2(k.numpy())
    wv, sv = c2.quantize_pack2(v.numpy())
    O, LSE = att.attention(q.numpy()[:, :, None], c2.dequantize2(wk, sk, 128), c2.dequantize2(wv, sv, 128),
                           scale, False, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, LSE[:, :, 0])
    assert qa.read_device_flags() == 0
