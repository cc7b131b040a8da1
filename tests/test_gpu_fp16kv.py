"""GPU parity of the comparison paths ("Quantized Cross-Attention ... In-SRAM
Dequantization" §5.2): the INT4 cache dequantized to fp16 (bit for bit
against oracle/baselines), attention over an fp16 cache (decode and prefill,
within the attention tolerance of the float64 oracle), and the two chained
(post-dequantization)."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, check_guards, guarded, require_gpu
from oracle import baselines as bl
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _filled_cache(qa, seed, B, Hkv, N, D):
    cache = qa.KvCache.contiguous(B, Hkv, N, D)
    k, v = wl.kv_block(seed, "k", B, Hkv, N, D), wl.kv_block(seed, "v", B, Hkv, N, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    return cache, k, v


@pytest.mark.parametrize("D,n", [(128, 300), (64, 77), (128, 1)])
def test_dequantize_matches_oracle_bits(D, n):
    qa = require_gpu()
    B, Hkv, cap = 2, 3, 320
    cache, _, _ = _filled_cache(qa, 61, B, Hkv, cap, D)
    # a saturated scale: 7 * 65504 overflows binary16 (+-inf), 1 * 65504 does not
    cache.k_scales[0, 0, 0] = 65504.0
    kb, k16 = guarded((B, Hkv, n, D), torch.float16)
    vb, v16 = guarded((B, Hkv, n, D), torch.float16)
    qa.dequantize_kv(cache, B, n, k16, v16)
    torch.cuda.synchronize()
    check_guards(kb, "k_out")
    check_guards(vb, "v_out")
    for t, (codes, scales) in ((k16, (cache.k_codes, cache.k_scales)), (v16, (cache.v_codes, cache.v_scales))):
        want = bl.dequantize_fp16(codes[:, :, :n].cpu().numpy(), scales[:, :, :n].cpu().numpy())
        assert np.array_equal(t.cpu().numpy().view(np.uint16), want.view(np.uint16))
    assert qa.read_device_flags() == 0


def test_dequantize_paged_matches_gathered_rows():
    qa = require_gpu()
    B, Hkv, D = 3, 8, 128
    lens, table, P = wl.paged_layout(62, B, 100, 400, 64)
    cache = qa.KvCache.paged(P, Hkv, D, torch.from_numpy(table))
    for b, L in enumerate(lens):
        sub = qa.KvCache(cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales, D, Hkv,
                         page_table=cache.page_table[b:b + 1], num_pages=P)
        qa.quantize_kv(wl.kv_block(62 + b, "k", 1, Hkv, int(L), D).cuda(),
                       wl.kv_block(62 + b, "v", 1, Hkv, int(L), D).cuda(), sub)
    n = int(lens.min())
    k16, _ = qa.dequantize_kv(cache, B, n)
    kc, ks = cache.k_codes.cpu().numpy(), cache.k_scales.cpu().numpy()
    for b in range(B):
        pages = table[b, : (n + 63) // 64]
        codes = kc[pages].transpose(1, 0, 2, 3).reshape(Hkv, -1, D // 2)[:, :n]
        scales = ks[pages].transpose(1, 0, 2).reshape(Hkv, -1)[:, :n]
        want = bl.dequantize_fp16(codes, scales)
        assert np.array_equal(k16[b].cpu().numpy().view(np.uint16), want.view(np.uint16))
    assert qa.read_device_flags() == 0


def _fp16_cache(seed, B, Hkv, cap, D, lens, poison=True):
    """fp16 K, V [B, Hkv, cap, D] with the rows past each length set to NaN
    (a kernel that reads them into its sums fails the comparison)."""
    k = wl.kv_block(seed, "k", B, Hkv, cap, D).half()
    v = wl.kv_block(seed, "v", B, Hkv, cap, D).half()
    if poison:
        for b, L in enumerate(lens):
            k[b, :, L:] = float("nan")
            v[b, :, L:] = float("nan")
    return k, v


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, lens, splits, scale
    (3, 16, 4, 128, [1000, 513, 77], 0, 1 / math.sqrt(128)),
    (3, 16, 4, 128, [1000, 513, 77], 1, 1 / math.sqrt(128)),
    (3, 16, 4, 128, [1000, 513, 77], 7, 1.0),
    (2, 4, 4, 64, [200, 0], 3, 0.125),          # G = 1, an empty sequence
    (1, 64, 8, 128, [4099], 0, 1 / math.sqrt(128)),
])
def test_decode_fp16_matches_oracle(case):
    qa = require_gpu()
    B, Hq, Hkv, D, lens, splits, scale = case
    cap = max(64, -(-max(lens) // 64) * 64)
    k, v = _fp16_cache(63, B, Hkv, cap, D, lens)
    q = wl.queries(63, B, Hq, D)
    ob, out = guarded((B, Hq, D), torch.float16)
    lb, lse = guarded((B, Hq), torch.float32)
    qa.decode_fp16(q.cuda(), k.cuda(), v.cuda(), torch.tensor(lens, dtype=torch.int32), max(lens), scale, splits,
                   out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    O, L = bl.attention_fp16(q.numpy()[:, :, None], np.nan_to_num(k.numpy()), np.nan_to_num(v.numpy()), scale,
                             False, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, L[:, :, 0])
    assert qa.read_device_flags() == 0


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, nq, nk, causal
    (2, 8, 2, 128, 300, 300, True),
    (1, 4, 4, 128, 100, 700, True),     # chunked: bottom-right causal
    (2, 6, 2, 64, 129, 257, False),
    (1, 2, 1, 128, 1, 1, True),
])
def test_prefill_fp16_matches_oracle(case):
    qa = require_gpu()
    B, Hq, Hkv, D, nq, nk, causal = case
    cap = -(-nk // 64) * 64 + 64
    k, v = _fp16_cache(64, B, Hkv, cap, D, [nk] * B)
    q = wl.queries(64, B, Hq, nq, D)
    scale = 1 / math.sqrt(D)
    ob, out = guarded((B, Hq, nq, D), torch.float16)
    lb, lse = guarded((B, Hq, nq), torch.float32)
    qa.prefill_fp16(q.cuda(), k.cuda(), v.cuda(), nk, scale, causal, out=out, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, "out")
    check_guards(lb, "lse")
    O, L = bl.attention_fp16(q.numpy(), k.numpy()[:, :, :nk], v.numpy()[:, :, :nk], scale, causal)
    assert_close_attention(out, O)
    assert_close_lse(lse, L)
    assert qa.read_device_flags() == 0


def test_post_dequant_decode_and_prefill_match_oracle():
    """Dequantize the INT4 cache to fp16 in HBM, then attend it: the oracle
    is attention over fl16(c * s)."""
    qa = require_gpu()
    B, Hq, Hkv, D, N = 2, 16, 4, 128, 700
    cache, _, _ = _filled_cache(qa, 65, B, Hkv, N, D)
    k16, v16 = qa.dequantize_kv(cache, B, cache.capacity)
    pk, sk = cache.k_codes.cpu().numpy(), cache.k_scales.cpu().numpy()
    pv, sv = cache.v_codes.cpu().numpy(), cache.v_scales.cpu().numpy()
    scale = 1 / math.sqrt(D)
    q = wl.queries(65, B, Hq, D)
    lens = [N, 333]
    out = qa.decode_fp16(q.cuda(), k16, v16, torch.tensor(lens, dtype=torch.int32), N, scale)
    O, _ = bl.attention_post_dequant(q.numpy()[:, :, None], pk, sk, pv, sv, scale, False, lens)
    assert_close_attention(out, O[:, :, 0])
    qp = wl.queries(66, B, Hq, 200, D)
    outp = qa.prefill_fp16(qp.cuda(), k16, v16, N, scale, True)
    Op, _ = bl.attention_post_dequant(qp.numpy(), pk[:, :, :N], sk[:, :, :N], pv[:, :, :N], sv[:, :, :N], scale, True)
    assert_close_attention(outp, Op)
    assert qa.read_device_flags() == 0
