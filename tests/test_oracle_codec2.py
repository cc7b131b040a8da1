"""Pins of the INT2 codec oracle (oracle/codec2.py): hand-derived vectors,
exact rational rounding, the bit positions of the sixteen-per-word packing,
invariants (TurboAttention, arXiv 2412.08585, §3.2: 2-bit heads)."""

from fractions import Fraction

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import codec2 as c2


def _rne(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def test_hand_vectors():
    x = np.array([[3.0, 0.0, -1.5, 1.5, -3.0, 0.5, -1.0, 2.0]], np.float32)
    c, s = c2.quantize_rows2(x)
    assert s.tolist() == [3.0]                        # absmax 3 -> s = 3
    # x / s = 1, 0, -1/2, 1/2, -1, 1/6, -1/3, 2/3; the ties go to 0 (even)
    assert c.tolist() == [[1, 0, 0, 0, -1, 0, 0, 1]]
    # absmax 0.1: s = fl16(fl32(0.1)) = 0.0999755859375
    assert c2.row_scales2(np.array([[0.1, 0.0]], np.float32)).tolist() == [0.0999755859375]
    assert c2.row_scales2(np.array([[1e6, 0.0]], np.float32)).tolist() == [65504.0]  # saturates
    assert c2.quantize_rows2(np.zeros((1, 4), np.float32))[0].tolist() == [[0, 0, 0, 0]]


def test_packing_bit_positions():
    codes = np.zeros((1, 32), np.int8)
    codes[0, :3] = [1, -1, 1]                         # 1 | 3 << 2 | 1 << 4
    assert c2.pack16(codes).tolist() == [[1 + (3 << 2) + (1 << 4), 0]]
    codes = np.zeros((1, 32), np.int8)
    codes[0, 31] = -1                                 # word 1, field 15: 0b11 << 30
    assert c2.pack16(codes).tolist() == [[0, 3 << 30]]
    w = c2.pack16(np.full((1, 128), -1, np.int8))     # D = 128: 8 words, 32 bytes
    assert w.shape == (1, 8) and all(int(v) == 0xFFFFFFFF for v in w[0])


def test_unpack_inverts_pack_for_every_field_value():
    rng = np.random.default_rng(5)
    c = rng.integers(-2, 2, size=(50, 128)).astype(np.int8)
    assert np.array_equal(c2.unpack16(c2.pack16(c), 128), c)
    c = rng.integers(-2, 2, size=(50, 40)).astype(np.int8)
    assert np.array_equal(c2.unpack16(c2.pack16(c), 40), c)


def test_rounding_equals_exact_rationals_and_invariants():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((200, 16)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    x[0, :4] = [2.0, 1.0, -1.0, 0.5]                  # exact ties at +-1/2
    c, s = c2.quantize_rows2(x)
    assert c[0, :4].tolist() == [1, 0, 0, 0]
    for r in range(x.shape[0]):
        sr = Fraction(float(s[r]))
        for j in range(x.shape[1]):
            want = max(-1, min(1, _rne(Fraction(float(x[r, j])) / sr)))
            assert int(c[r, j]) == want
        assert np.abs(c[r]).max() == 1                # the absmax maps to +-1
        err = np.abs(x[r].astype(np.float64) - c[r] * float(s[r]))
        assert err.max() <= float(s[r]) / 2 + 1e-12 * float(s[r])
    assert np.abs(c).max() <= 1


def test_dequantize_hand_vector():
    words = c2.pack16(np.array([[1, 0, -1, 1, 0, -1]], np.int8))
    got = c2.dequantize2(words, np.array([0.5], np.float16), 6)
    assert got.tolist() == [[0.5, 0.0, -0.5, 0.5, 0.0, -0.5]]


MUTATIONS = [
    ("row_scales2", "am / np.float32(QMAX2)", "am / np.float32(2)"),              # wrong divisor
    ("quantize_rows2", "np.rint(q)", "np.floor(q + 0.5)"),                      # ties away from even
    ("pack16", "c & 3", "c & 1"),                                                # field mask
    ("pack16", "shifts = 2 * np.arange", "shifts = 3 * np.arange"),              # field width
    ("unpack16", "f - 4", "f - 2"),                                              # sign extension
    ("dequantize2", "unpack16(words, d).astype(np.float64) *", "unpack16(words, d).astype(np.float64) + 0 *"),  # scale dropped
]
PINS = [test_hand_vectors, test_packing_bit_positions, test_unpack_inverts_pack_for_every_field_value,
        test_rounding_equals_exact_rationals_and_invariants, test_dequantize_hand_vector]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] + ":" + m[2] for m in MUTATIONS])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    func, old, new = mutation
    assert mutant_fails_a_pin(monkeypatch, c2, func, old, new, PINS), mutation
