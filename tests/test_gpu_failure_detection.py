"""Failure detection on the GPU without faulting it: a bounded wait that is
made to run out (an mbarrier nothing arrives at) returns with
QATTN_FLAG_WAIT_TIMEOUT, and the context stays usable afterwards."""

import math

import pytest
import torch

from common import assert_close_attention, require_gpu
from oracle import attention as att
from oracle import codec
from quantized_kv_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_a_timeout():
    qa = require_gpu()
    assert qa.read_device_flags() == 0
    for limit in (1000, 2_000_000):  # ~0.5 us and ~1 ms at 2 GHz
        assert qa.check_wait_timeout(limit) == qa.FLAG_WAIT_TIMEOUT
    # the library's own status word is untouched
    assert qa.read_device_flags() == 0


def test_context_usable_after_the_timeout_check():
    qa = require_gpu()
    assert qa.check_wait_timeout(100_000) == qa.FLAG_WAIT_TIMEOUT
    B, Hq, Hkv, D, L = 1, 4, 2, 128, 300
    k = wl.kv_block(7, "k", B, Hkv, L, D)
    v = wl.kv_block(7, "v", B, Hkv, L, D)
    q = wl.queries(7, B, Hq, D)
    cache = qa.KvCache.contiguous(B, Hkv, 320, D)
    qa.quantize_kv(k.cuda(), v.cuda(), cache)
    out = qa.decode(q.cuda(), cache, torch.tensor([L], dtype=torch.int32).cuda(), L, 1 / math.sqrt(D), 2)
    pk, sk = codec.quantize_pack(k.numpy())
    pv, sv = codec.quantize_pack(v.numpy())
    O, _ = att.attention_quantized(q.numpy()[:, :, None, :], pk, sk, pv, sv, 1 / math.sqrt(D), False)
    assert_close_attention(out, O[:, :, 0, :])
    assert qa.read_device_flags() == 0
