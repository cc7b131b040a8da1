"""GPU parity of qattn_quantize_kv: codes and scales bit-exact against the oracle."""

import os

import numpy as np
import pytest
import torch

from common import require_gpu
from oracle import attention as att
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _golden_rows(golden_dir, d):
    rows = []
    with open(os.path.join(golden_dir, "codec_vectors.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                xs = [float.fromhex(v) for v in line.split("|")[0].split()]
                row = np.zeros(d, np.float32)
                row[: len(xs)] = xs
                rows.append(row)
    return np.stack(rows)


def _readback(cache):
    return (cache.k_codes.cpu().numpy(), cache.k_scales.cpu().numpy(),
            cache.v_codes.cpu().numpy(), cache.v_scales.cpu().numpy())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_contiguous_append_bit_exact(d, dtype, golden_dir):
    qa = require_gpu()
    B, H, n, cap = 3, 2, 150, 256
    k = wl.kv_block(11, "k", B, H, n, d, wl.outlier_channels(11, H, d, 4), 10.0)
    v = wl.kv_block(11, "v", B, H, n, d)
    g = torch.from_numpy(_golden_rows(golden_dir, d))       # ties, saturation, subnormal scales
    k[0, 0, : g.shape[0]] = g
    v[1, 1, : g.shape[0]] = -g
    k[2, 1, 7] = 0.0                                          # all-zero row
    k, v = k.to(dtype), v.to(dtype)
    cache = qa.KvCache.contiguous(B, H, cap, d)
    start = torch.tensor([0, 10, 120], dtype=torch.int32)    # last sequence runs past capacity
    qa.quantize_kv(k.cuda(), v.cuda(), cache, start.cuda())
    kc, ks, vc, vs = _readback(cache)
    for name, x, cc, ss in (("k", k, kc, ks), ("v", v, vc, vs)):
        pk, sk = codec.quantize_pack(x.float().numpy())
        for b in range(B):
            p0 = int(start[b])
            m = min(n, cap - p0)
            assert (cc[b, :, p0:p0 + m] == pk[b, :, :m]).all(), (name, b)
            assert (ss[b, :, p0:p0 + m].view(np.uint16) == sk[b, :, :m].view(np.uint16)).all(), (name, b)
            assert (cc[b, :, :p0] == 0).all() and (cc[b, :, p0 + m:] == 0).all()   # nothing else written
    assert qa.read_device_flags() == 0


def test_paged_append_bit_exact():
    qa = require_gpu()
    d, H = 128, 4
    lens, table, P = wl.paged_layout(5, 6, 1, 300, 64)
    cache = qa.KvCache.paged(P, H, d, torch.from_numpy(table))
    ref = {}
    for b, n in enumerate(lens):
        k = wl.kv_slice(5, "k", b, 0, int(n) * H, d).reshape(1, H, int(n), d)
        v = wl.kv_slice(5, "v", b, 0, int(n) * H, d).reshape(1, H, int(n), d)
        sub = qa.KvCache(cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales, d, H,
                         page_table=cache.page_table[b:b + 1], num_pages=P)
        # append in two pieces to exercise start_pos with paging
        h1 = int(n) // 3
        qa.quantize_kv(k[:, :, :h1].cuda(), v[:, :, :h1].cuda(), sub)
        qa.quantize_kv(k[:, :, h1:].cuda(), v[:, :, h1:].cuda(), sub, torch.tensor([h1], dtype=torch.int32).cuda())
        ref[b] = (codec.quantize_pack(k.numpy()[0]), codec.quantize_pack(v.numpy()[0]))
    kc, ks, vc, vs = _readback(cache)
    gk, gks = att.gather_pages(kc, ks, table, lens, 64)
    gv, gvs = att.gather_pages(vc, vs, table, lens, 64)
    for b, n in enumerate(lens):
        (pk, sk), (pv, sv) = ref[b]
        assert (gk[b, :, :n] == pk).all() and (gks[b, :, :n].view(np.uint16) == sk.view(np.uint16)).all()
        assert (gv[b, :, :n] == pv).all() and (gvs[b, :, :n].view(np.uint16) == sv.view(np.uint16)).all()
    # nothing else written: pool rows past each sequence's length (its last
    # page's tail) and pages no table row names keep their zeros
    used = np.zeros(ks.shape, dtype=bool)  # [P, H, 64]
    for b, n in enumerate(lens):
        for t in range(int(n)):
            used[table[b, t // 64], :, t % 64] = True
    for name, a in (("k codes", kc), ("v codes", vc)):
        assert (a[~used] == 0).all(), name
    for name, a in (("k scales", ks), ("v scales", vs)):
        assert (a[~used].view(np.uint16) == 0).all(), name
    assert qa.read_device_flags() == 0


def test_missing_page_is_skipped_and_flagged():
    qa = require_gpu()
    d, H = 64, 1
    table = torch.tensor([[0, -1]], dtype=torch.int32)
    cache = qa.KvCache.paged(1, H, d, table)
    k = torch.randn(1, H, 128, d)
    qa.quantize_kv(k.cuda(), k.cuda(), cache)
    assert qa.read_device_flags() & qa.FLAG_BAD_PAGE
    pk, sk = codec.quantize_pack(k.numpy()[0, :, :64])
    assert (cache.k_codes.cpu().numpy()[0] == pk).all()
    assert qa.read_device_flags() == 0                        # cleared by the previous read
