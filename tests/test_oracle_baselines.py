"""Pins of oracle/baselines.py (the FP16 and post-dequantization comparison
paths of "Quantized Cross-Attention ... In-SRAM Dequantization" §5.2) against
values fixed by IEEE binary16 rounding and by the attention definition."""

import os
import struct

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import attention as att
from oracle import baselines as bl
from oracle import codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant_fp16_vectors.txt")


def _vectors():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, s, want, _ = [x.strip() for x in line.split("|", 3)]
        out.append((int(c), int(s, 16), int(want, 16)))
    return out


def _packed(codes):
    """Pack codes (even count) as the cache stores them."""
    return codec.pack_nibbles(np.asarray(codes, dtype=np.int8))


@pytest.mark.parametrize("c,sbits,want", _vectors())
def test_dequantize_fp16_hand_vectors(c, sbits, want):
    packed = _packed([c, 0])
    s = np.array([sbits], dtype=np.uint16).view(np.float16)
    got = bl.dequantize_fp16(packed[None], s)[0, 0]
    assert int(np.asarray(got).view(np.uint16)) == want


def test_dequantize_fp16_matches_an_independent_binary16_rounding():
    """Every code against every finite positive fp16 scale: numpy's float16
    cast agrees with CPython's own binary16 packing (struct 'e', a separate
    implementation of the same IEEE rounding) of the exact product; products
    beyond the binary16 range are the infinities IEEE rounding gives."""
    scales = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16)
    for c in range(-7, 8):
        packed = np.broadcast_to(_packed([c, 0]), (scales.size, 1))
        got = bl.dequantize_fp16(packed, scales)[:, 0].view(np.uint16)
        exact = c * scales.astype(np.float64)
        for i in range(0, scales.size, 97):       # a spread sample of all 31743 scales
            try:
                want = struct.unpack("<H", struct.pack("<e", float(exact[i])))[0]
            except OverflowError:
                want = 0x7C00 if exact[i] > 0 else 0xFC00
            assert got[i] == want, (c, hex(int(scales[i:i + 1].view(np.uint16)[0])))


def test_dequantize_fp16_half_ulp_bound_and_exact_codes():
    """|fl16(cs) - cs| <= half an fp16 ulp of cs; codes 0, +-1, +-2, +-4 times
    a normal scale need at most 11 significant bits, so they are exact."""
    rng = np.random.default_rng(0)
    s = rng.uniform(2.0**-10, 2.0**8, 20000).astype(np.float16)
    for c in range(-7, 8):
        packed = np.broadcast_to(_packed([c, 0]), (s.size, 1))
        got = bl.dequantize_fp16(packed, s)[:, 0].astype(np.float64)
        exact = c * s.astype(np.float64)
        mag = np.maximum(np.abs(exact), 2.0**-14)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 10)
        assert (np.abs(got - exact) <= ulp / 2).all()
        if abs(c) in (0, 1, 2, 4):
            assert (got == exact).all()


def test_post_dequant_equals_fused_when_products_are_fp16_exact():
    """With power-of-two scales every c*s is an fp16 value, so attending the
    FP16 copy is attending the exact dequantized cache."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, N, D = 2, 4, 2, 37, 16
    codes = rng.integers(-7, 8, (B, Hkv, N, D))
    k_p = codec.pack_nibbles(codes.astype(np.int8))
    v_p = codec.pack_nibbles(rng.integers(-7, 8, (B, Hkv, N, D)).astype(np.int8))
    k_s = (2.0 ** rng.integers(-6, 2, (B, Hkv, N))).astype(np.float16)
    v_s = (2.0 ** rng.integers(-6, 2, (B, Hkv, N))).astype(np.float16)
    q = rng.standard_normal((B, Hq, 3, D)).astype(np.float16)
    O1, L1 = bl.attention_post_dequant(q, k_p, k_s, v_p, v_s, 0.3, True)
    O2, L2 = att.attention_quantized(q, k_p, k_s, v_p, v_s, 0.3, True)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_post_dequant_uses_the_rounded_copy():
    """A scale whose products round: the post-dequant result is attention over
    the rounded values, and differs from the exact-dequant result."""
    D = 8
    codes = np.array([[[[7, 5, 3, 6, 7, 5, 3, 6]] * 4]], dtype=np.int8)   # [1, 1, 4, 8]
    k_p = codec.pack_nibbles(codes)
    s = np.full((1, 1, 4), np.array([0x3C02], dtype=np.uint16).view(np.float16)[0])
    x16 = bl.dequantize_fp16(k_p, s)
    assert x16.dtype == np.float16
    assert float(x16[0, 0, 0, 1]) == 5.0078125                  # the tie of the golden vectors
    q = np.ones((1, 1, 1, D), dtype=np.float16)
    O_pd, _ = bl.attention_post_dequant(q, k_p, s, k_p, s, 1.0)
    O_ref, _ = att.attention(q, x16.astype(np.float64), x16.astype(np.float64), 1.0)
    O_ex, _ = att.attention_quantized(q, k_p, s, k_p, s, 1.0)
    assert np.array_equal(O_pd, O_ref)
    assert not np.array_equal(O_pd, O_ex)


def test_attention_fp16_is_the_plain_definition_on_fp16_values():
    """Single key: O is that key's value row; two identical keys: their mean."""
    v = np.array([[[[0.5, -1.25, 3.0, 2.0], [0.5, -1.25, 3.0, 2.0]]]], dtype=np.float16)
    k = np.array([[[[1.0, 2.0, 0.0, -1.0], [1.0, 2.0, 0.0, -1.0]]]], dtype=np.float16)
    q = np.array([[[[0.25, 0.5, 1.0, 2.0]]]], dtype=np.float16)
    O, L = bl.attention_fp16(q, k[:, :, :1], v[:, :, :1], 0.5)
    assert np.array_equal(O[0, 0, 0], v[0, 0, 0].astype(np.float64))
    assert L[0, 0, 0] == pytest.approx(0.5 * (0.25 + 1.0 - 2.0))
    O2, L2 = bl.attention_fp16(q, k, v, 0.5)
    assert np.allclose(O2[0, 0, 0], v[0, 0, 0].astype(np.float64), rtol=0, atol=1e-15)
    assert L2[0, 0, 0] == pytest.approx(0.5 * (0.25 + 1.0 - 2.0) + np.log(2.0))


def _all_hand_vectors():
    for args in _vectors():
        test_dequantize_fp16_hand_vectors(*args)


MUTATIONS = [
    ("dequantize_fp16", "exact.astype(np.float16)", "(exact * (1 + 2.0**-30)).astype(np.float16)"),  # ties away from zero
    ("dequantize_fp16", "codec.dequantize(packed, scales)", "codec.dequantize(packed, scales) * 1.0009765625"),  # off by an ulp
    ("attention_fp16", "np.asarray(v16, dtype=np.float16)", "np.asarray(k16, dtype=np.float16)"),   # K used as V
    ("attention_fp16", "softmax_scale, causal", "1.0, causal"),                                       # scale dropped
    ("attention_post_dequant", "dequantize_fp16(v_packed, v_scales)", "dequantize_fp16(v_packed, k_scales)"),  # K scales on V
    ("attention_post_dequant", "softmax_scale, causal, k_lens)", "softmax_scale, False, k_lens)"),     # mask dropped
]
PINS = [_all_hand_vectors, test_dequantize_fp16_half_ulp_bound_and_exact_codes,
        test_post_dequant_equals_fused_when_products_are_fp16_exact, test_post_dequant_uses_the_rounded_copy,
        test_attention_fp16_is_the_plain_definition_on_fp16_values]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] + ":" + m[2][:40] for m in MUTATIONS])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    func, old, new = mutation
    assert mutant_fails_a_pin(monkeypatch, bl, func, old, new, PINS), mutation
