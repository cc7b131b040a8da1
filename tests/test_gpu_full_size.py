"""GPU parity at the bench's full sizes and launch configurations, on sampled
outputs the float64 oracle computes one slice at a time.

The whole workload runs on the GPU exactly as the bench times it (split
count, CTA layout); the oracle regenerates the sampled (sequence, kv-head)
slices from the same seeded generators, checks their codes and scales bit
for bit, and recomputes the sampled rows of O and lse.
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


def _fill(qa, seed, B, Hkv, N, D, oc=None, oscale=1.0):
    cache = qa.KvCache.contiguous(B, Hkv, N, D)
    for b in range(B):
        k = torch.stack([wl.kv_slice(seed, "k", b, h, N, D, oc, oscale) for h in range(Hkv)])[None]
        v = torch.stack([wl.kv_slice(seed, "v", b, h, N, D) for h in range(Hkv)])[None]
        sub = qa.KvCache(cache.k_codes[b:b + 1], cache.k_scales[b:b + 1], cache.v_codes[b:b + 1],
                         cache.v_scales[b:b + 1], D, Hkv, capacity=cache.capacity)
        qa.quantize_kv(k.cuda(), v.cuda(), sub)
    torch.cuda.synchronize()
    return cache


def _oracle_slice(qa, cache, seed, b, h, N, D, oc=None, oscale=1.0):
    """Oracle codes of one (sequence, kv-head) slice, checked against the cache."""
    k = wl.kv_slice(seed, "k", b, h, N, D, oc, oscale).numpy()
    v = wl.kv_slice(seed, "v", b, h, N, D).numpy()
    pk, sk = codec.quantize_pack(k)
    pv, sv = codec.quantize_pack(v)
    assert np.array_equal(cache.k_codes[b, h, :N].cpu().numpy(), pk)
    assert np.array_equal(cache.v_codes[b, h, :N].cpu().numpy(), pv)
    assert np.array_equal(cache.k_scales[b, h, :N].cpu().numpy().view(np.uint16), sk.view(np.uint16))
    assert np.array_equal(cache.v_scales[b, h, :N].cpu().numpy().view(np.uint16), sv.view(np.uint16))
    return pk, sk, pv, sv


def _decode_full(name, samples, splits):
    qa = require_gpu()
    cfg = wl.WORKLOADS[name]
    B, Hq, Hkv, D, N, seed = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Nk"], cfg["seed"]
    G = Hq // Hkv
    oc = wl.outlier_channels(seed, Hkv, D, cfg["outliers"]) if cfg.get("outliers") else None
    oscale = cfg.get("outlier_scale", 1.0)
    cache = _fill(qa, seed, B, Hkv, N, D, oc, oscale)
    q = wl.queries(seed, B, Hq, D)
    scale = 1 / math.sqrt(D)
    lens = torch.full((B,), N, dtype=torch.int32)
    out, lse = qa.decode(q.cuda(), cache, lens.cuda(), N, scale, splits, return_lse=True)
    for b, h in samples:
        pk, sk, pv, sv = _oracle_slice(qa, cache, seed, b, h, N, D, oc, oscale)
        qs = q.numpy()[b:b + 1, h * G:(h + 1) * G, None, :]
        O, L = att.attention_quantized(qs, pk[None, None], sk[None, None], pv[None, None], sv[None, None],
                                       scale, False)
        assert_close_attention(out[b:b + 1, h * G:(h + 1) * G], O[:, :, 0])
        assert_close_lse(lse[b:b + 1, h * G:(h + 1) * G], L[:, :, 0])
    assert qa.read_device_flags() == 0


def test_long_context_decode_full_size():
    """B=1, Hq=64, Hkv=8, D=128, Nk=131072, 152 splits (the bench's launch)."""
    _decode_full("long_decode", [(0, 5)], 152)


def test_batched_gqa_decode_full_size():
    """B=8, Hq=32, Hkv=8, D=128, Nk=4096, outlier channels, automatic splits."""
    _decode_full("gqa_decode", [(0, 0), (3, 4), (7, 7)], 0)


def test_causal_prefill_full_size():
    """B=2, Hq=32, Hkv=8, D=128, Nq=Nk=8192, causal: sampled rows of two heads
    of two (sequence, kv-head) slices, first and last rows of the blocks included."""
    qa = require_gpu()
    cfg = wl.WORKLOADS["causal_prefill"]
    B, Hq, Hkv, D, N, seed = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Nk"], cfg["seed"]
    G = Hq // Hkv
    cache = _fill(qa, seed, B, Hkv, N, D)
    q = wl.queries(seed, B, Hq, N, D)
    scale = 1 / math.sqrt(D)
    out, lse = qa.prefill(q.cuda(), cache, N, scale, True, return_lse=True)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 129, 4095, 4096, 8064, 8190, 8191],
                                     rng.integers(0, N, 22)]))
    for b, h in [(0, 0), (1, 6)]:
        pk, sk, pv, sv = _oracle_slice(qa, cache, seed, b, h, N, D)
        k_hat = codec.dequantize(pk, sk)
        v_hat = codec.dequantize(pv, sv)
        for hq in (h * G, h * G + G - 1):
            qh = q.numpy()[b, hq].astype(np.float64)
            O = np.zeros((len(rows), D))
            L = np.zeros(len(rows))
            for i, r in enumerate(rows):  # row r sees keys 0..r (bottom-right causal, Nq = Nk)
                o, lv = att.attention(qh[None, None, r:r + 1], k_hat[None, None, :r + 1], v_hat[None, None, :r + 1],
                                      scale, False)
                O[i], L[i] = o[0, 0, 0], lv[0, 0, 0]
            idx = torch.as_tensor(rows, device=out.device)
            assert_close_attention(out[b, hq].index_select(0, idx), O)
            assert_close_lse(lse[b, hq].index_select(0, idx), L)
    assert qa.read_device_flags() == 0


def _paged_rows(cache, table, b, h, n):
    """Rows 0..n-1 of (sequence b, kv-head h) gathered from the page pool."""
    pages = torch.as_tensor(table[b, : (n + 63) // 64].astype(np.int64), device=cache.k_codes.device)
    kc = cache.k_codes.index_select(0, pages)[:, h].reshape(-1, cache.k_codes.shape[-1])[:n]
    vc = cache.v_codes.index_select(0, pages)[:, h].reshape(-1, cache.v_codes.shape[-1])[:n]
    ks = cache.k_scales.index_select(0, pages)[:, h].reshape(-1)[:n]
    vs = cache.v_scales.index_select(0, pages)[:, h].reshape(-1)[:n]
    return kc.cpu().numpy(), ks.cpu().numpy(), vc.cpu().numpy(), vs.cpu().numpy()


@pytest.mark.parametrize("scale", [1 / math.sqrt(128), 1.0])
def test_paged_varlen_decode_full_size(scale):
    """64 sequences with lengths uniform in [512, 32768], 64-token pages in a
    randomly permuted pool, Hq=32, Hkv=8, D=128, automatic splits, one
    qattn_decode_append step (the bench's launch), at softmax scale 1/sqrt(128)
    and 1.0.  Three sequences (the shortest, the longest and one more) hold the
    oracle's seeded rows and are checked whole: codes and scales bit for bit,
    every q-head's O and lse.  The others hold device-drawn rows of the same
    distribution (seeded), which keeps the workload's size and raggedness; for
    them the check is that every output is finite."""
    qa = require_gpu()
    cfg = wl.WORKLOADS["paged_decode"]
    B, Hq, Hkv, D, seed = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["seed"]
    G = Hq // Hkv
    lens, table, P = wl.paged_layout(seed, B, cfg["len_lo"], cfg["len_hi"], cfg["page"])
    assert (lens >= cfg["len_lo"]).all() and (lens <= cfg["len_hi"]).all()
    cache = qa.KvCache.paged(P, Hkv, D, torch.from_numpy(table))
    picked = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 17})
    g = torch.Generator(device="cuda")
    k_new = torch.empty(B, Hkv, D, device="cuda")
    v_new = torch.empty(B, Hkv, D, device="cuda")
    for b, n in enumerate(lens):
        n = int(n)
        if b in picked:
            k = torch.stack([wl.kv_slice(seed, "k", b, h, n, D) for h in range(Hkv)])[None].cuda()
            v = torch.stack([wl.kv_slice(seed, "v", b, h, n, D) for h in range(Hkv)])[None].cuda()
        else:
            g.manual_seed(seed * 7919 + b)
            k = torch.randn(1, Hkv, n, D, device="cuda", generator=g)
            v = torch.randn(1, Hkv, n, D, device="cuda", generator=g)
        sub = qa.KvCache(cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales, D, Hkv,
                         page_table=cache.page_table[b:b + 1], num_pages=P)
        qa.quantize_kv(k[:, :, : n - 1], v[:, :, : n - 1], sub)   # the cached rows
        k_new[b], v_new[b] = k[0, :, n - 1], v[0, :, n - 1]        # the step appends the last one
        del k, v
    q = wl.queries(seed, B, Hq, D)
    sl = torch.from_numpy(lens.astype(np.int32)).cuda()
    out, lse = qa.decode_append(q.cuda(), k_new, v_new, cache, sl, int(cfg["len_hi"]), scale, 0, return_lse=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    for b in picked:
        n = int(lens[b])
        for h in range(Hkv):
            k = wl.kv_slice(seed, "k", b, h, n, D).numpy()
            v = wl.kv_slice(seed, "v", b, h, n, D).numpy()
            pk, sk = codec.quantize_pack(k)
            pv, sv = codec.quantize_pack(v)
            kc, ks, vc, vs = _paged_rows(cache, table, b, h, n)
            assert np.array_equal(kc, pk) and np.array_equal(vc, pv)
            assert np.array_equal(ks.view(np.uint16), sk.view(np.uint16))
            assert np.array_equal(vs.view(np.uint16), sv.view(np.uint16))
            qs = q.numpy()[b:b + 1, h * G:(h + 1) * G, None, :]
            O, L = att.attention_quantized(qs, pk[None, None], sk[None, None], pv[None, None], sv[None, None],
                                           scale, False)
            assert_close_attention(out[b:b + 1, h * G:(h + 1) * G], O[:, :, 0])
            assert_close_lse(lse[b:b + 1, h * G:(h + 1) * G], L[:, :, 0])
    assert qa.read_device_flags() == 0
