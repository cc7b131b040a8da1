"""GPU parity of the segment-cluster decode: one thread-block cluster of S CTAs
per (sequence, kv-head group) segment, whose partials are merged through
distributed shared memory inside the decode kernel (qattn_decode_plan reports
cluster = S; no merge kernel, no partials in global memory).

The shapes are sized so that a 152-SM GB300 takes that path (clusters of 2 and
4, the 8- and 12-warp layouts, D = 128 and 64, ragged lengths with an empty
sequence and one-token sequences).  Each case checks that the plan is a
cluster plan, that qattn_decode_append writes the new rows bit-exact and
equals the two-call form (append, then qattn_decode) bit for bit, that the
cost-balanced path (an explicit split count) agrees to the parity tolerance,
and O and lse against the float64 oracle.
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

CASES = [
    # B, Hq, Hkv, D, lens (after the append)
    (8, 32, 8, 128, [4096, 1, 0, 300, 256, 257, 2048, 3333]),  # S = 2: empty, one-token, row first in a stage
    (4, 32, 8, 128, [3000, 1500, 64, 2500]),                    # S = 4
    (8, 64, 8, 64, [2000, 77, 1024, 1999, 5, 640, 1500, 2000]),  # D = 64, 8 q-heads a kv-head
    (8, 32, 8, 64, [11000, 10999, 384, 385, 11000, 1, 7000, 11000]),  # the 12-warp layout
]


def _cluster_plan(qa, B, Hq, Hkv, D, L):
    plan = qa.decode_plan(B, Hq, Hkv, D, L)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms < 128:
        pytest.skip(f"{sms} SMs: these shapes were sized for a GB300")
    assert plan["cluster"] >= 2, plan
    assert plan["ctas"] == B * Hkv * plan["cluster"], plan
    return plan


@pytest.mark.parametrize("case", CASES)
def test_cluster_decode_append(case):
    qa = require_gpu()
    B, Hq, Hkv, D, lens = case
    L = max(lens)
    plan = _cluster_plan(qa, B, Hq, Hkv, D, L)
    seed = 31
    cap = max(64, -(-L // 64) * 64)
    k, v = wl.kv_block(seed, "k", B, Hkv, L, D), wl.kv_block(seed, "v", B, Hkv, L, D)
    q = wl.queries(seed, B, Hq, D)
    scale = 1 / math.sqrt(D)
    a = qa.KvCache.contiguous(B, Hkv, cap, D)
    qa.quantize_kv(k.cuda(), v.cuda(), a)
    for b, n in enumerate(lens):  # the new rows must come from the append
        if n > 0:
            for t in (a.k_codes, a.v_codes, a.k_scales, a.v_scales):
                t[b, :, n - 1] = 0
    c = qa.KvCache(a.k_codes.clone(), a.k_scales.clone(), a.v_codes.clone(), a.v_scales.clone(), D, Hkv, capacity=cap)
    idx = torch.tensor([max(n - 1, 0) for n in lens])
    k_new = k[torch.arange(B), :, idx].contiguous()
    v_new = v[torch.arange(B), :, idx].contiguous()
    sl = torch.tensor(lens, dtype=torch.int32).cuda()
    out, lse = qa.decode_append(q.cuda(), k_new.cuda(), v_new.cuda(), a, sl, L, scale, 0, return_lse=True)
    # the two-call form takes the same cluster path: bit for bit
    qa.quantize_kv(k_new[:, :, None].cuda(), v_new[:, :, None].cuda(), c,
                   torch.tensor([n - 1 if n > 0 else cap for n in lens], dtype=torch.int32).cuda())
    out2, lse2 = qa.decode(q.cuda(), c, sl, L, scale, 0, return_lse=True)
    # the cost-balanced ranges and the merge kernel (an explicit split count)
    out3, lse3 = qa.decode(q.cuda(), c, sl, L, scale, plan["ctas"], return_lse=True)
    torch.cuda.synchronize()
    for x, y in ((a.k_codes, c.k_codes), (a.v_codes, c.v_codes), (a.k_scales, c.k_scales), (a.v_scales, c.v_scales)):
        assert torch.equal(x, y)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert_close_attention(out, out3.float().cpu().numpy().astype(np.float64), "cluster vs cost-balanced",
                           max_abs=2e-3, mean_abs=2e-4)
    # the oracle on the whole history
    kh, vh = k.clone(), v.clone()
    for b, n in enumerate(lens):
        if n > 0:
            kh[b, :, n - 1], vh[b, :, n - 1] = k_new[b], v_new[b]
    pk, sk = codec.quantize_pack(kh.numpy())
    pv, sv = codec.quantize_pack(vh.numpy())
    for b, n in enumerate(lens):
        if n > 0:
            assert np.array_equal(a.k_codes[b, :, n - 1].cpu().numpy(), pk[b, :, n - 1])
            assert np.array_equal(a.v_scales[b, :, n - 1].cpu().numpy().view(np.uint16),
                                  sv[b, :, n - 1].view(np.uint16))
    O, LSE = att.attention_quantized(q.numpy()[:, :, None], pk, sk, pv, sv, scale, False, lens)
    assert_close_attention(out, O[:, :, 0])
    assert_close_lse(lse, LSE[:, :, 0])
    empty = [b for b, n in enumerate(lens) if n == 0]
    for b in empty:  # a sequence with no key: O = 0, lse = -inf
        assert torch.count_nonzero(out[b]) == 0
        assert torch.isneginf(lse[b]).all()
    assert qa.read_device_flags() == 0


def test_plan_paths():
    """Which path the plan names for shapes outside the cluster rule."""
    qa = require_gpu()
    if torch.cuda.get_device_properties(0).multi_processor_count < 128:
        pytest.skip("sized for a GB300")
    # an explicit split count, a paged pool, INT3, a listed cache: the cost-balanced ranges
    assert qa.decode_plan(8, 32, 8, 128, 4096, num_splits=152)["cluster"] == 0
    assert qa.decode_plan(8, 32, 8, 128, 4096, paged=True)["cluster"] == 0
    assert qa.decode_plan(8, 32, 8, 128, 4096, code_bits=3)["cluster"] == 0
    assert qa.decode_plan(8, 32, 8, 128, 4096, listed=True)["cluster"] == 0
    # one sequence of one stage: nothing to split
    assert qa.decode_plan(1, 1, 1, 64, 256)["cluster"] == 0
    # too few segments to fill the SMs with clusters of at most 16 CTAs
    assert qa.decode_plan(1, 8, 1, 128, 100000)["cluster"] == 0
