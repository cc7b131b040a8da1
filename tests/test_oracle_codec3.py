"""Pins of the INT3 codec oracle (oracle/codec3.py): hand-derived vectors,
exact rational rounding, bit positions of the ten-per-word packing
("Quantized Cross-Attention ... In-SRAM Dequantization" §3.3), invariants."""

from fractions import Fraction

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import codec3 as c3


def _rne(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def test_hand_vectors():
    x = np.array([[3.0, 0.0, -1.5, 1.5, -3.0, 0.5, -0.5, 2.5, 1.0, -2.0]], np.float32)
    c, s = c3.quantize_rows3(x)
    assert s.tolist() == [1.0]                        # absmax 3 -> s = 1
    assert c.tolist() == [[3, 0, -2, 2, -3, 0, 0, 2, 1, -2]]   # ties to even
    # absmax 1: s = fl16(1/3) = 1365/1024 * 2^-2
    assert c3.row_scales3(np.array([[1.0, 0.0]], np.float32)).tolist() == [0.333251953125]
    assert c3.row_scales3(np.array([[1e6, 0.0]], np.float32)).tolist() == [65504.0]  # saturates


def test_packing_bit_positions():
    codes = np.zeros((1, 20), np.int8)
    codes[0, :3] = [1, -1, 3]                         # 1 | 7 << 3 | 3 << 6
    assert c3.pack10(codes).tolist() == [[1 + (7 << 3) + (3 << 6), 0]]
    codes = np.zeros((1, 20), np.int8)
    codes[0, 19] = -2                                 # word 1, field 9: 0b110 << 27
    assert c3.pack10(codes).tolist() == [[0, 6 << 27]]
    # D = 128: 13 words, elements 120..127 in bits 0..23 of word 12, the rest zero
    w = c3.pack10(np.full((1, 128), -1, np.int8))
    assert w.shape == (1, 13)
    assert all(int(v) == (1 << 30) - 1 for v in w[0, :12])
    assert int(w[0, 12]) == (1 << 24) - 1


def test_unpack_inverts_pack_for_every_field_value():
    rng = np.random.default_rng(3)
    c = rng.integers(-4, 4, size=(50, 128)).astype(np.int8)
    assert np.array_equal(c3.unpack10(c3.pack10(c), 128), c)
    c = rng.integers(-4, 4, size=(50, 64)).astype(np.int8)
    assert np.array_equal(c3.unpack10(c3.pack10(c), 64), c)


def test_rounding_equals_exact_rationals_and_invariants():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((200, 16)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    c, s = c3.quantize_rows3(x)
    for r in range(x.shape[0]):
        sr = Fraction(float(s[r]))
        for j in range(x.shape[1]):
            want = max(-3, min(3, _rne(Fraction(float(x[r, j])) / sr)))
            assert int(c[r, j]) == want
        assert np.abs(c[r]).max() == 3                # the absmax maps to +-3
        err = np.abs(x[r].astype(np.float64) - c[r] * float(s[r]))
        assert err.max() <= float(s[r]) / 2 + 1e-12 * float(s[r])
    assert np.abs(c).max() <= 3


def test_dequantize_hand_vector():
    words = c3.pack10(np.array([[3, 0, -1, -3, 2, 1, 0, -2, 1, 3, -1]], np.int8))
    got = c3.dequantize3(words, np.array([0.25], np.float16), 11)
    assert got.tolist() == [[0.75, 0.0, -0.25, -0.75, 0.5, 0.25, 0.0, -0.5, 0.25, 0.75, -0.25]]


MUTATIONS = [
    ("row_scales3", "am / np.float32(QMAX3)", "am / np.float32(4)"),              # wrong divisor
    ("quantize_rows3", "np.rint(q)", "np.floor(q + 0.5)"),                      # ties away from even
    ("pack10", "c & 7", "c & 3"),                                                # field mask
    ("pack10", "shifts = 3 * np.arange", "shifts = 4 * np.arange"),              # field width
    ("unpack10", "f - 8", "f - 4"),                                              # sign extension
    ("dequantize3", "unpack10(words, d).astype(np.float64) *", "unpack10(words, d).astype(np.float64) + 0 *"),  # scale dropped
]
PINS = [test_hand_vectors, test_packing_bit_positions, test_unpack_inverts_pack_for_every_field_value,
        test_rounding_equals_exact_rationals_and_invariants, test_dequantize_hand_vector]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] + ":" + m[2] for m in MUTATIONS])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    func, old, new = mutation
    assert mutant_fails_a_pin(monkeypatch, c3, func, old, new, PINS), mutation
