"""qattn_decode_noalloc, called through the C ABI.

This entry point is for callers that cannot allocate device memory (a plugin
handed only its input and output buffers, or a device whose memory a caching
allocator has already reserved): it runs the split-KV decode with its
partials in a fixed device array the library owns.  It launches the same
kernels with the same split count as qattn_decode, so its output must equal
qattn_decode's bit for bit, call after call (a partial overwrite of the
shared array would show up as a difference), and sizes whose partials do not
fit that array must be refused before any work.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

from common import require_gpu
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 * 1024 * 1024


def _contiguous(qa, seed, B, Hq, Hkv, D, lens):
    L = max(lens)
    cache = qa.KvCache.contiguous(B, Hkv, L, D)
    qa.quantize_kv(wl.kv_block(seed, "k", B, Hkv, L, D).cuda(), wl.kv_block(seed, "v", B, Hkv, L, D).cuda(), cache)
    return cache, wl.queries(seed, B, Hq, D).cuda(), torch.tensor(lens, dtype=torch.int32).cuda(), L


def _listed(qa, seed, B, Hq, Hkv, D, lens):
    """The 4-bit cache of a headwise plan with two 2-bit heads: it lists 6 of
    the model's 8 kv-heads, so its scratch is sized by the model's heads."""
    L = max(lens)
    k, v = wl.kv_block(seed, "k", B, Hkv, L, D).cuda(), wl.kv_block(seed, "v", B, Hkv, L, D).cuda()
    bits = [4] * Hkv
    bits[1] = bits[5] = 2
    four, _ = qa.mixed_caches(bits, B, L, D)
    qa.quantize_kv(k, v, four)
    return four, wl.queries(seed, B, Hq, D).cuda(), torch.tensor(lens, dtype=torch.int32).cuda(), L


def _paged(qa, seed, B, Hq, Hkv, D, lo, hi):
    lens, table, P = wl.paged_layout(seed, B, lo, hi, 64)
    cache = qa.KvCache.paged(P, Hkv, D, torch.from_numpy(table))
    for b, n in enumerate(lens):
        sub = qa.KvCache(cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales, D, Hkv,
                         page_table=cache.page_table[b:b + 1], num_pages=P)
        qa.quantize_kv(wl.kv_block(seed + b, "k", 1, Hkv, int(n), D).cuda(),
                       wl.kv_block(seed + b, "v", 1, Hkv, int(n), D).cuda(), sub)
    return cache, wl.queries(seed, B, Hq, D).cuda(), torch.from_numpy(lens.astype(np.int32)).cuda(), int(hi)


def _noalloc(qa, q, cache, sl, L, scale, splits, out, lse):
    lib = qa.load_library()
    B, Hq, D = q.shape
    st = cache.struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = lib.qattn_decode_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.byref(st),
                                      ctypes.c_void_p(sl.data_ptr()), B, Hq, L, scale, splits,
                                      ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)
    assert status == qa.QATTN_OK, lib.qattn_last_error().decode()
    torch.cuda.synchronize()


CASES = [  # (name, builder, args, splits): every case cuts sequences into several ranges
    ("contiguous_d128", _contiguous, (51, 3, 16, 4, 128, [1000, 513, 77]), 0),
    ("contiguous_d64", _contiguous, (52, 2, 8, 8, 64, [2048, 3]), 7),
    ("listed_cache", _listed, (53, 2, 32, 8, 128, [900, 1500]), 0),
    ("paged", _paged, (54, 5, 32, 8, 128, 1, 2000), 9),
]


@pytest.mark.parametrize("name,builder,args,splits", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_decode_on_consecutive_calls(name, builder, args, splits):
    qa = require_gpu()
    cache, q, sl, L = builder(qa, *args)
    B, Hq, D = q.shape
    assert 0 < qa.decode_workspace_size(B, Hq, cache.workspace_kv_heads, D, L, splits) <= SCRATCH_BYTES
    scale = 1 / math.sqrt(D)
    # a listed cache writes only its own heads' rows: start both outputs equal
    ref = torch.zeros_like(q)
    ref_lse = torch.zeros(B, Hq, dtype=torch.float32, device=q.device)
    qa.decode(q, cache, sl, L, scale, splits, out=ref, lse=ref_lse)
    for _ in range(2):  # the second call finds the first call's partials in the array
        out = torch.zeros_like(q)
        lse = torch.zeros(B, Hq, dtype=torch.float32, device=q.device)
        _noalloc(qa, q, cache, sl, L, scale, splits, out, lse)
        assert torch.equal(out, ref)
        assert torch.equal(lse, ref_lse)
    assert torch.isfinite(ref.float()).all()
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
