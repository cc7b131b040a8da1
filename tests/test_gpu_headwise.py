"""GPU parity of headwise mixed 2/4-bit precision (TurboAttention, arXiv
2412.08585, §3.2) against oracle/headwise: the plan's priorities and bits
exactly (binary64 in channel order on both sides), and a decode over the two
caches of a plan (4-bit heads, 2-bit heads, each listing its model heads)
against float64 attention over the head-by-head dequantized values."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, require_gpu
from oracle import headwise as hw
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _prompt(seed, B, H, n, D=128, spread=None):
    k = wl.kv_block(seed, "k", B, H, n, D)
    v = wl.kv_block(seed, "v", B, H, n, D)
    if spread is not None:  # per-head scale, so the heads' priorities differ widely
        s = torch.tensor(spread, dtype=torch.float32)[None, :, None, None]
        k, v = k * s, v * s
    return k, v


@pytest.mark.parametrize("dt", [torch.float32, torch.float16])
@pytest.mark.parametrize("case", [
    # B, Hkv, n, lens, num_low, D
    (2, 8, 300, [300, 123], 3, 128),
    (3, 4, 64, [0, 64, 1], 1, 64),
    (1, 8, 1000, None, 8, 128),
    (2, 6, 40, [0, 0], 2, 128),        # no rows: every priority 0, the first heads go to 2 bits
])
def test_plan_matches_oracle_exactly(case, dt):
    qa = require_gpu()
    B, H, n, lens, low, D = case
    k, v = _prompt(5, B, H, n, D, spread=[0.5 + 0.25 * h for h in range(H)])
    k, v = k.to(dt), v.to(dt)
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    bits, prio = qa.headwise_plan(k.cuda(), v.cuda(), low, None if ln is None else ln.cuda())
    want_p = hw.priorities(k.float().numpy(), v.float().numpy(), lens)
    assert np.array_equal(prio.cpu().numpy(), want_p)
    assert np.array_equal(bits.cpu().numpy(), hw.plan_bits(want_p, low))


def test_plan_ties_go_to_the_lower_head():
    qa = require_gpu()
    k, v = _prompt(9, 1, 1, 50)
    k, v = k.repeat(1, 5, 1, 1), v.repeat(1, 5, 1, 1)   # five identical heads
    bits, prio = qa.headwise_plan(k.cuda(), v.cuda(), 2)
    assert len(set(prio.cpu().tolist())) == 1
    assert bits.cpu().tolist() == [2, 2, 4, 4, 4]


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, lens, num_low, splits, scale
    (2, 16, 8, [700, 333], 3, 0, 1 / math.sqrt(128)),
    (3, 8, 4, [0, 64, 900], 2, 5, 1 / math.sqrt(128)),   # empty sequence, ragged tails
    (1, 32, 8, [4096], 4, 64, 1 / math.sqrt(128)),       # many splits
    (2, 16, 4, [500, 257], 1, 3, 1.0),                   # G = 4, softmax scale 1.0
    (2, 8, 4, [300, 200], 0, 0, 0.1),                    # every head at 4 bits (one cache)
    (2, 8, 4, [300, 200], 4, 0, 0.1),                    # every head at 2 bits (one cache)
])
def test_mixed_decode(case):
    qa = require_gpu()
    B, Hq, Hkv, lens, low, splits, scale = case
    L = max(max(lens), 1)
    k, v = _prompt(11, B, Hkv, L, spread=[0.4 + 0.3 * ((5 * h) % Hkv) for h in range(Hkv)])
    bits, _ = qa.headwise_plan(k.cuda(), v.cuda(), low, torch.tensor(lens, dtype=torch.int32).cuda())
    caches = qa.mixed_caches(bits, B, max(64, -(-L // 64) * 64), 128)
    for c in caches:
        if c is not None:
            qa.quantize_kv(k.cuda(), v.cuda(), c)   # each cache stores its own heads
    q = wl.queries(11, B, Hq, 128)
    out, lse = qa.decode_mixed(q.cuda(), caches, torch.tensor(lens, dtype=torch.int32).cuda(), L, scale, splits,
                               return_lse=True)
    O, LSE = hw.attention_mixed(q.numpy()[:, :, None], k.numpy(), v.numpy(), bits.cpu().numpy(), scale, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, LSE[:, :, 0])
    assert qa.read_device_flags() == 0


def test_listed_cache_writes_only_its_heads_and_flags_a_bad_index():
    qa = require_gpu()
    B, Hq, Hkv, L = 2, 8, 4, 200
    k, v = _prompt(13, B, Hkv, L)
    cache = qa.KvCache.contiguous(B, 2, 256, 128)
    cache.kv_head_index = torch.tensor([3, 1], dtype=torch.int32, device="cuda")
    cache.model_kv_heads = Hkv
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    q = wl.queries(13, B, Hq, 128)
    out = torch.full((B, Hq, 128), 7.0, dtype=torch.float16, device="cuda")
    qa.decode(q.cuda(), cache, torch.tensor([200, 150], dtype=torch.int32).cuda(), L, 0.1, 0, out=out)
    O, _ = hw.attention_mixed(q.numpy()[:, :, None], k.numpy(), v.numpy(), [4] * Hkv, 0.1, [200, 150])
    o = out.cpu()
    for h in range(Hkv):
        rows = o[:, 2 * h:2 * h + 2]
        if h in (3, 1):
            assert_close_attention(rows, O[:, 2 * h:2 * h + 2, 0])
        else:
            assert torch.all(rows == 7.0)                # not this cache's heads: untouched
    assert qa.read_device_flags() == 0
    cache.kv_head_index = torch.tensor([3, 9], dtype=torch.int32, device="cuda")  # 9: no such head
    out2 = out.clone()
    qa.decode(q.cuda(), cache, torch.tensor([200, 150], dtype=torch.int32).cuda(), L, 0.1, 0, out=out2)
    assert qa.read_device_flags() & qa.FLAG_BAD_HEAD
    assert torch.equal(out2[:, 6:8], out[:, 6:8])         # head 3 still attended
