"""qattn_decode_noalloc, called through the C ABI.

This entry point is for callers that cannot allocate device memory (a plugin
handed only its input and output buffers, or a device whose memory a caching
allocator has already reserved): it runs the split-KV decode with its
partials in a fixed device array the library owns.  Its output must match
qattn_decode's, call after call, and sizes whose partials do not fit that
array must be refused before any work.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes
import math

import pytest
import torch

from common import LSE_ABS, O_MAX_ABS, require_gpu
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 * 1024 * 1024


def _case(qa, seed, B, Hq, Hkv, D, lens):
    L = max(lens)
    cache = qa.KvCache.contiguous(B, Hkv, L, D)
    qa.quantize_kv(wl.kv_block(seed, "k", B, Hkv, L, D).cuda(), wl.kv_block(seed, "v", B, Hkv, L, D).cuda(), cache)
    q = wl.queries(seed, B, Hq, D).cuda()
    sl = torch.tensor(lens, dtype=torch.int32).cuda()
    return cache, q, sl, L


def _noalloc(qa, q, cache, sl, L, scale, splits):
    lib = qa.load_library()
    B, Hq, D = q.shape
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=q.device)
    st = cache.struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = lib.qattn_decode_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.byref(st),
                                      ctypes.c_void_p(sl.data_ptr()), B, Hq, L, scale, splits,
                                      ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)
    assert status == qa.QATTN_OK, lib.qattn_last_error().decode()
    torch.cuda.synchronize()
    return out, lse


def test_noalloc_matches_decode_on_consecutive_calls():
    qa = require_gpu()
    cases = [  # (seed, B, Hq, Hkv, D, lens, splits): both use more than one split
        (51, 3, 16, 4, 128, [1000, 513, 77], 0),
        (52, 2, 8, 8, 64, [2048, 3], 7),
    ]
    for seed, B, Hq, Hkv, D, lens, splits in cases:
        cache, q, sl, L = _case(qa, seed, B, Hq, Hkv, D, lens)
        assert 0 < qa.decode_workspace_size(B, Hq, Hkv, D, L, splits) <= SCRATCH_BYTES
        scale = 1 / math.sqrt(D)
        ref, ref_lse = qa.decode(q, cache, sl, L, scale, splits, return_lse=True)
        out, lse = _noalloc(qa, q, cache, sl, L, scale, splits)
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        assert (out.float() - ref.float()).abs().max().item() <= O_MAX_ABS
        assert (lse - ref_lse).abs().max().item() <= LSE_ABS
    assert qa.read_device_flags() == 0


def test_noalloc_refuses_sizes_beyond_its_scratch():
    qa = require_gpu()
    lib = qa.load_library()
    B, Hq, Hkv, D, L, splits = 1, 64, 8, 128, 131072, 1024
    assert qa.decode_workspace_size(B, Hq, Hkv, D, L, splits) > SCRATCH_BYTES
    fake = 0x10000  # never dereferenced: the size check comes first
    st = qa.KvCacheStruct()
    st.k_codes = st.k_scales = st.v_codes = st.v_scales = fake
    st.head_dim, st.num_kv_heads, st.capacity = D, Hkv, L
    status = lib.qattn_decode_noalloc(fake, ctypes.byref(st), fake, B, Hq, L, 1.0, splits, fake, None, None)
    assert status == qa.QATTN_ERR_UNSUPPORTED
    assert b"static scratch" in lib.qattn_last_error()
