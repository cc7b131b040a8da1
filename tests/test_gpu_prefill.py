"""GPU parity of qattn_prefill (causal and not, chunked Nq < Nk) against the oracle."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, require_gpu
from oracle import attention as att
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run_prefill(seed, B, Hq, Hkv, D, nq, nk, causal, scale, cap=None):
    qa = require_gpu()
    cap = cap or max(64, -(-nk // 64) * 64)
    k = wl.kv_block(seed, "k", B, Hkv, nk, D)
    v = wl.kv_block(seed, "v", B, Hkv, nk, D)
    q = wl.queries(seed, B, Hq, nq, D)
    cache = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    out, lse = qa.prefill(q.cuda(), cache, nk, scale, causal, return_lse=True)
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, L = att.attention_quantized(q.numpy(), pk, sk, pv, sv, scale, causal)
    assert_close_attention(out, O)
    assert_close_lse(lse, L)
    assert qa.read_device_flags() == 0


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, nq, nk, causal
    (2, 4, 2, 128, 300, 300, True),     # ragged q and k tails, several tiles
    (2, 4, 2, 128, 300, 300, False),
    (1, 2, 1, 128, 77, 300, True),      # chunked prefill: bottom-right causal
    (1, 8, 2, 64, 200, 200, True),      # D = 64
    (1, 2, 2, 128, 1, 129, True),       # one query row
    (1, 2, 1, 128, 64, 64, True),       # exactly one tile
    (1, 4, 1, 128, 257, 513, False),
])
def test_prefill(case):
    B, Hq, Hkv, D, nq, nk, causal = case
    run_prefill(31, B, Hq, Hkv, D, nq, nk, causal, 1 / math.sqrt(D))


def test_prefill_scale_one():
    run_prefill(37, 1, 2, 1, 128, 130, 130, True, 1.0)


def test_prefill_row_equals_decode():
    """A causal prefill row i equals a decode of that query over keys <= i."""
    qa = require_gpu()
    B, Hq, Hkv, D, N = 1, 4, 2, 128, 200
    k = wl.kv_block(41, "k", B, Hkv, N, D)
    v = wl.kv_block(41, "v", B, Hkv, N, D)
    q = wl.queries(41, B, Hq, N, D).cuda()
    cache = qa.KvCache.contiguous(B, Hkv, N, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    out = qa.prefill(q, cache, N, 0.1, True)
    for i in (0, 63, 64, 130, 199):
        od = qa.decode(q[:, :, i].contiguous(), cache, torch.tensor([i + 1], dtype=torch.int32).cuda(), N, 0.1, 1)
        assert (od.float() - out[:, :, i].float()).abs().max().item() <= 2e-3


@pytest.mark.parametrize("nq,causal", [(100, True), (300, True), (77, False)])
def test_prefill_paged(nq, causal):
    """Chunked prefill of a paged cache: pages of each sequence scattered over
    a randomly permuted pool, the last page row of the table unused (-1)."""
    qa = require_gpu()
    B, Hq, Hkv, D, nk, page = 2, 8, 2, 128, 300, 64
    npg = -(-nk // page)
    perm = torch.randperm(B * npg, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    table = torch.full((B, npg + 1), -1, dtype=torch.int32)
    table[:, :npg] = perm.view(B, npg)
    cache = qa.KvCache.paged(B * npg, Hkv, D, table)
    k = wl.kv_block(43, "k", B, Hkv, nk, D)
    v = wl.kv_block(43, "v", B, Hkv, nk, D)
    for b in range(B):
        sub = qa.KvCache(cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales, D, Hkv,
                         page_table=cache.page_table[b:b + 1], num_pages=B * npg)
        qa.quantize_kv(k[b:b + 1].cuda(), v[b:b + 1].cuda(), sub)
    q = wl.queries(43, B, Hq, nq, D)
    scale = 1 / math.sqrt(D)
    out, lse = qa.prefill(q.cuda(), cache, nk, scale, causal, return_lse=True)
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, L = att.attention_quantized(q.numpy(), pk, sk, pv, sv, scale, causal)
    assert_close_attention(out, O)
    assert_close_lse(lse, L)
    assert qa.read_device_flags() == 0
