"""Pins of the headwise mixed-precision oracle (oracle/headwise.py):
TurboAttention (arXiv 2412.08585) §3.2's gap and std statistics, checked by
hand, against an exact-rational standard deviation, and by invariants; the
selection of the lowest-priority heads; the head-by-head composition of the
mixed-precision attention."""

import math
import statistics

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import attention as att
from oracle import codec, codec2
from oracle import headwise as hw


def test_priority_by_hand():
    # channel gaps 2 and 4 (mean 3, population std 1); overall gap 5 - 0
    assert hw.head_priority(np.array([[0.0, 1.0], [2.0, 5.0]], np.float32)) == 5.0
    # one row: every channel gap is 0, so std = 0 whatever the overall gap
    assert hw.head_priority(np.array([[1.0, -1.0, 0.0, 3.0]], np.float32)) == 0.0
    # gaps 1, 1, 4, 2 (mean 2, variance 1.5); overall gap 4 - (-1)
    x = np.array([[0, -1, 0, 1], [1, 0, 4, 3]], np.float32)
    assert hw.head_priority(x) == 5.0 * math.sqrt(1.5)
    assert hw.head_priority(np.zeros((0, 8), np.float32)) == 0.0


def test_priority_against_independent_statistics():
    rng = np.random.default_rng(2)
    for _ in range(20):
        x = (rng.standard_normal((37, 16)) * rng.uniform(0.1, 9)).astype(np.float32)
        gaps = [float(x[:, j].max()) - float(x[:, j].min()) for j in range(16)]
        gap = max(float(v) for v in x.ravel()) - min(float(v) for v in x.ravel())
        want = gap * statistics.pstdev(gaps)          # exact-rational mean and variance
        assert math.isclose(hw.head_priority(x), want, rel_tol=1e-13)


def test_priority_invariants():
    rng = np.random.default_rng(4)
    x = rng.integers(-50, 50, size=(30, 8)).astype(np.float32)
    p = hw.head_priority(x)
    assert hw.head_priority(x + 7.0) == p             # a shift moves no gap
    assert hw.head_priority(4.0 * x) == 16.0 * p      # gap and std both scale
    assert hw.head_priority(x[::-1]) == p             # row order
    assert hw.head_priority(x[:, ::-1]) == p          # channel order (integer sums are exact)
    wide = x.copy()
    wide[:, 0] *= 3.0                                 # one channel spreads: std and priority grow
    assert hw.head_priority(wide) > p


def test_plan_bits_and_key_value_maximum():
    assert hw.plan_bits([3.0, 1.0, 2.0, 1.0], 2).tolist() == [4, 2, 4, 2]
    assert hw.plan_bits([1.0, 1.0, 1.0], 1).tolist() == [2, 4, 4]   # ties: lower head first
    assert hw.plan_bits([5.0, 1.0], 0).tolist() == [4, 4]
    assert hw.plan_bits([5.0, 1.0], 2).tolist() == [2, 2]
    # 64 heads in two priority classes: the 20 low ones are the first 20 of the lower class
    want = [2 if h % 2 == 0 and h < 40 else 4 for h in range(64)]
    assert hw.plan_bits([1.0, 2.0] * 32, 20).tolist() == want
    rng = np.random.default_rng(6)
    k = rng.standard_normal((2, 3, 10, 8)).astype(np.float32)
    v = rng.standard_normal((2, 3, 10, 8)).astype(np.float32)
    k[:, 0] *= 10.0                                   # head 0: keys dominate
    v[:, 2] *= 10.0                                   # head 2: values dominate
    p = hw.priorities(k, v)
    for h in range(3):
        kr = np.concatenate([k[b, h] for b in range(2)])
        vr = np.concatenate([v[b, h] for b in range(2)])
        assert p[h] == max(hw.head_priority(kr), hw.head_priority(vr))
    assert hw.plan_bits(p, 1).tolist() == [4, 2, 4]
    # ragged lengths: rows past lens[b] do not count
    k2 = k.copy()
    k2[0, :, 7:] = 1e4
    assert np.array_equal(hw.priorities(k2, v, [7, 10]), hw.priorities(k, v, [7, 10]))


def test_mixed_attention_composes_head_by_head():
    rng = np.random.default_rng(8)
    B, Hkv, G, N, D = 2, 3, 2, 40, 16
    q = rng.standard_normal((B, Hkv * G, 1, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, N, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, N, D)).astype(np.float32)
    o4, l4 = hw.attention_mixed(q, k, v, [4, 4, 4], 0.25)
    p, s = codec.quantize_pack(k)
    pv, sv = codec.quantize_pack(v)
    oq, lq = att.attention_quantized(q, p, s, pv, sv, 0.25)
    assert np.array_equal(o4, oq) and np.array_equal(l4, lq)
    w, s2 = codec2.quantize_pack2(k)
    wv, sv2 = codec2.quantize_pack2(v)
    o2, l2 = att.attention(q, codec2.dequantize2(w, s2, D), codec2.dequantize2(wv, sv2, D), 0.25)
    assert np.array_equal(hw.attention_mixed(q, k, v, [2, 2, 2], 0.25)[0], o2)
    om, lm = hw.attention_mixed(q, k, v, [2, 4, 2], 0.25)
    for h in range(Hkv):
        src_o, src_l = (o2, l2) if h != 1 else (o4, l4)
        assert np.array_equal(om[:, h * G:(h + 1) * G], src_o[:, h * G:(h + 1) * G])
        assert np.array_equal(lm[:, h * G:(h + 1) * G], src_l[:, h * G:(h + 1) * G])
    # 2-bit heads lose accuracy against the unquantized values, 4-bit ones less
    of, _ = att.attention(q, k, v, 0.25)
    assert np.abs(o2 - of).mean() > np.abs(o4 - of).mean()


MUTATIONS = [
    ("head_priority", "math.sqrt(sq / d)", "math.sqrt(sq / (d - 1))"),                 # sample, not population std
    ("head_priority", "float(mx.max()) - float(mn.min())", "float(mx.max()) - float(mx.min())"),  # wrong gap
    ("head_priority", "return gap * math.sqrt", "return gap + math.sqrt"),              # sum, not product
    ("priorities", "max(head_priority(kr), head_priority(vr))", "head_priority(kr)"),  # values ignored
    ("priorities", "k[b, h, :ln[b]]", "k[b, h]"),                                        # lengths ignored
    ("plan_bits", "bits[order[:n_low]] = 2", "bits[order[len(bits) - n_low:]] = 2"),    # highest go low
    ("plan_bits", 'kind="stable"', 'kind="quicksort"'),                                  # ties unordered
    ("dequantize_mixed", "if b == 2:", "if b != 2:"),                                    # widths swapped
]
PINS = [test_priority_by_hand, test_priority_against_independent_statistics, test_priority_invariants,
        test_plan_bits_and_key_value_maximum, test_mixed_attention_composes_head_by_head]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] + ":" + m[2] for m in MUTATIONS])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    func, old, new = mutation
    assert mutant_fails_a_pin(monkeypatch, hw, func, old, new, PINS), mutation
