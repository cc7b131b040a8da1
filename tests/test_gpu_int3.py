"""GPU parity of the INT3 cache ("Quantized Cross-Attention ... In-SRAM
Dequantization" §3.3: ten 3-bit values per 32-bit word) against oracle/codec3:
the append's words and scales bit for bit, and split-KV decode over the INT3
rows against float64 attention over their dequantized values."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, check_guards, guarded, require_gpu
from oracle import attention as att
from oracle import codec3 as c3
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _words(t):
    """uint8 [..., 52] -> little-endian uint32 [..., 13]."""
    return t.cpu().numpy().view(np.uint32)


def _fill(qa, seed, B, Hkv, L, D=128, dt=torch.float32):
    cap = max(64, -(-L // 64) * 64)
    k = wl.kv_block(seed, "k", B, Hkv, L, D)
    v = wl.kv_block(seed, "v", B, Hkv, L, D)
    cache = qa.KvCache.contiguous(B, Hkv, cap, D, code_bits=3)
    qa.quantize_kv(k.to(dt).cuda(), v.to(dt).cuda(), cache)
    torch.cuda.synchronize()
    return cache, k.to(dt).float(), v.to(dt).float()


@pytest.mark.parametrize("dt", [torch.float32, torch.float16])
def test_int3_append_is_bit_exact(dt):
    qa = require_gpu()
    cache, k, v = _fill(qa, 61, 2, 3, 200, dt=dt)
    for x, codes, scales in ((k, cache.k_codes, cache.k_scales), (v, cache.v_codes, cache.v_scales)):
        w, s = c3.quantize_pack3(x.numpy())
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
def test_int3_decode(case):
    qa = require_gpu()
    B, Hq, Hkv, lens, splits, scale = case
    L = max(max(lens), 1)
    cache, k, v = _fill(qa, 67, B, Hkv, L)
    q = wl.queries(67, B, Hq, 128)
    ob, out = guarded((B, Hq, 128), torch.float16)
    lb, lse = guarded((B, Hq), torch.float32)
    qa.decode(q.cuda(), cache, torch.tensor(lens, dtype=torch.int32).cuda(), L, scale, splits, out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    wk, sk = c3.quantize_pack3(k.numpy())
    wv, sv = c3.quantize_pack3(v.numpy())
    O, LSE = att.attention(q.numpy()[:, :, None], c3.dequantize3(wk, sk, 128), c3.dequantize3(wv, sv, 128),
                           scale, False, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, LSE[:, :, 0])
    assert qa.read_device_flags() == 0
