"""Decode at the library's limits, against the float64 oracle: the largest batch
(QATTN_MAX_BATCH sequences, ragged and empty lengths, the per-sequence arrays
the decode keeps in shared memory at their largest), the fused append at that
batch, and the largest split count (QATTN_MAX_SPLITS ranges over one long
sequence: most ranges hold no stage, so the merge's empty-range path runs)."""

import math

import numpy as np
import pytest
import torch

from common import assert_close_attention, assert_close_lse, require_gpu
from oracle import attention as att
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_BATCH = 1024
MAX_SPLITS = 1024


def _sample(lens):
    """Sequences the oracle checks: every 16th, plus every empty one and every one at
    the capacity (the kernels run all of them)."""
    hi = max(lens)
    return sorted(set(range(0, len(lens), 16)) | {b for b, n in enumerate(lens) if n in (0, hi)})


def _oracle(q, k, v, lens, scale, idx):
    pk, sk = codec.quantize_pack(k.numpy()[idx])
    pv, sv = codec.quantize_pack(v.numpy()[idx])
    O, LSE = att.attention_quantized(q.numpy()[idx][:, :, None], pk, sk, pv, sv, scale, False, [lens[b] for b in idx])
    return O[:, :, 0], LSE[:, :, 0], pk, sv


def _lens(seed, B, hi):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, hi + 1, size=B)
    lens[::97] = 0       # some empty sequences
    lens[5::89] = hi     # some at the capacity
    return [int(x) for x in lens]


@pytest.mark.parametrize("splits", [0, 300])
def test_decode_at_max_batch(splits):
    qa = require_gpu()
    B, Hq, Hkv, D, cap = MAX_BATCH, 8, 2, 128, 192
    lens = _lens(81, B, cap)
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(81, "k", B, Hkv, cap, D), wl.kv_block(81, "v", B, Hkv, cap, D)
    q = wl.queries(81, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    out, lse = qa.decode(q.cuda(), cache, torch.tensor(lens, dtype=torch.int32).cuda(), cap, scale, splits,
                         return_lse=True)
    idx = _sample(lens)
    O, LSE, _, _ = _oracle(q, k, v, lens, scale, idx)
    assert_close_attention(out[idx], O)
    assert_close_lse(lse[idx], LSE)
    assert qa.read_device_flags() == 0


def test_decode_append_at_max_batch():
    qa = require_gpu()
    B, Hq, Hkv, D, cap = MAX_BATCH, 8, 2, 64, 128
    lens = [max(n, 1) for n in _lens(82, B, cap)]  # after the append every sequence has its new row
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(82, "k", B, Hkv, cap, D), wl.kv_block(82, "v", B, Hkv, cap, D)
    q = wl.queries(82, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    idx = torch.tensor([n - 1 for n in lens])
    k_new = (k[torch.arange(B), :, idx] * -0.75).contiguous()
    v_new = (v[torch.arange(B), :, idx] * -0.75).contiguous()
    out, lse = qa.decode_append(q.cuda(), k_new.cuda(), v_new.cuda(), cache, torch.tensor(lens, dtype=torch.int32).cuda(),
                                cap, scale, 0, return_lse=True)
    kh, vh = k.clone(), v.clone()
    for b, n in enumerate(lens):
        kh[b, :, n - 1], vh[b, :, n - 1] = k_new[b], v_new[b]
    idx = _sample(lens)
    O, LSE, pk, sv = _oracle(q, kh, vh, lens, scale, idx)
    for j, b in enumerate(idx):  # the appended rows, bit for bit
        n = lens[b]
        assert np.array_equal(cache.k_codes[b, :, n - 1].cpu().numpy(), pk[j, :, n - 1])
        assert np.array_equal(cache.v_scales[b, :, n - 1].cpu().numpy().view(np.uint16), sv[j, :, n - 1].view(np.uint16))
    assert_close_attention(out[idx], O)
    assert_close_lse(lse[idx], LSE)
    assert qa.read_device_flags() == 0


@pytest.mark.parametrize("n", [5000, 70000])
def test_decode_at_max_splits(n):
    qa = require_gpu()
    B, Hq, Hkv, D = 1, 8, 1, 128
    scale = 1 / math.sqrt(D)
    k, v = wl.kv_block(83, "k", B, Hkv, n, D), wl.kv_block(83, "v", B, Hkv, n, D)
    q = wl.queries(83, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, n, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    out, lse = qa.decode(q.cuda(), cache, torch.tensor([n], dtype=torch.int32).cuda(), n, scale, MAX_SPLITS,
                         return_lse=True)
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, LSE = att.attention_quantized(q.numpy()[:, :, None], pk, sk, pv, sv, scale, False, [n])
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, LSE[:, :, 0])
    assert qa.read_device_flags() == 0
