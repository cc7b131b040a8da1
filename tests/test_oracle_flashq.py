"""Pins of the decode-buffer oracle (oracle/flashq.py) against exact arithmetic
and closed forms: the universal scale, int8 rounding and clamping, the range
taken from the cached history, a flush that must reproduce representable rows,
and attention over a single buffered key.  TurboAttention (arXiv 2412.08585)
§3.3 (decoding buffer, universal scale, clamping) and §3.2 (8-bit symmetric
quantization)."""

from fractions import Fraction

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import codec
from oracle import flashq as fq


def _rne(fr: Fraction) -> int:
    """Round half to even of an exact rational."""
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def test_universal_scale_closed_forms():
    assert fq.universal_scale(127.0) == np.float16(1.0)
    assert fq.universal_scale(0.0) == np.float16(0.0)
    assert fq.universal_scale(254.0) == np.float16(2.0)
    # 1/127 = 0.0078740157...: binary16 keeps 10 fraction bits at 2^-7, 1032/1024 * 2^-7
    assert fq.universal_scale(1.0) == np.float16(0.00787353515625)
    assert fq.universal_scale(1e9) == np.float16(65504.0)  # saturates


def test_int8_codes_equal_exact_rounding_and_clamp():
    rng = np.random.default_rng(5)
    for u in (np.float16(1.0), np.float16(0.0371), np.float16(3.5), np.float16(6.1e-5)):
        x = (rng.standard_normal(400) * float(u) * 60).astype(np.float32)
        x[:4] = np.float32(float(u)) * np.array([2.5, -2.5, 3.5, 126.5], dtype=np.float32)  # ties
        c = fq.quantize_int8(x[None], np.asarray([u]))[0]
        for xi, ci in zip(x, c):
            want = _rne(Fraction(float(xi)) / Fraction(float(u)))
            assert int(ci) == max(-127, min(127, want)), (float(xi), float(u))
    c = fq.quantize_int8(np.array([[2.5, -2.5, 3.5, -0.5, 0.5, 1.5]], dtype=np.float32), np.asarray([np.float16(1)]))
    assert c.tolist() == [[2, -2, 4, 0, 0, 2]]
    big = fq.quantize_int8(np.array([[1000.0, -1000.0, 127.4]], dtype=np.float32), np.asarray([np.float16(1)]))
    assert big.tolist() == [[127, -127, 127]]                    # outliers clamp
    assert fq.quantize_int8(np.ones((1, 8), np.float32), np.asarray([np.float16(0)])).tolist() == [[0] * 8]


def test_history_range_is_seven_times_the_largest_scale():
    rows = np.zeros((3, 8), np.float32)
    rows[0, 0], rows[1, 3], rows[2, 5] = 14.0, -3.5, 0.25         # absmax 14 -> s = 2
    _, s = codec.quantize_pack(rows)
    assert float(fq.history_range(s)) == 14.0
    head = fq.BufferedHead(rows)
    assert float(head.r) == 14.0
    assert head.u == fq.universal_scale(14.0)
    assert float(fq.history_range(np.zeros(0, np.float16))) == 0.0


def test_first_row_sets_the_range_of_an_empty_history():
    head = fq.BufferedHead(np.zeros((0, 8), np.float32))
    row = np.array([127.0, -64.0, 3.0, 0.0, 1.0, -127.0, 5.0, 2.0], np.float32)
    c = head.append(row)
    assert head.u == np.float16(1.0) and c.tolist() == row.astype(int).tolist()


def test_outlier_past_the_range_is_clamped():
    head = fq.BufferedHead(np.array([[7.0, 0, 0, 0]], np.float32))  # R = 7
    c = head.append(np.array([70.0, -70.0, 3.5, 0.0], np.float32))
    u = float(fq.universal_scale(7.0))
    assert c[0] == 127 and c[1] == -127
    assert c[2] == _rne(Fraction(3.5) / Fraction(u))


def test_flush_reproduces_representable_rows():
    # buffered values c4 * s with |c4| <= 7 and one +-7 per row are INT4 rows: the
    # flush must give back exactly c4 and s; u = 1 keeps x~ = c8 exact
    head = fq.BufferedHead(np.array([[127.0] + [0.0] * 7], np.float32))  # R = 126.98... -> u = 1
    rng = np.random.default_rng(9)
    c4 = rng.integers(-7, 8, size=(fq.NB, 8))
    c4[:, 0] = 7 * np.where(rng.random(fq.NB) < 0.5, 1, -1)
    s = 2.0 ** rng.integers(0, 4, size=fq.NB)                           # 1, 2, 4, 8
    for row in c4 * s[:, None]:
        head.append(row.astype(np.float32))
    p, sc = head.flush()
    assert np.array_equal(sc.astype(np.float64), s)
    assert np.array_equal(codec.unpack_nibbles(p), c4)
    # the history row's INT4 scale is fl16(127 / 7) = 1161/1024 * 16 = 18.140625, so
    # R = 7 * 18.140625 = 126.984375 (and u = fl16(R / 127) = 1.0); the flushed rows'
    # 7 * max s = 56 does not raise it
    assert float(head.r) == max(126.984375, 7.0 * s.max())
    assert head.codes == []


def test_attention_over_one_buffered_key_is_its_value():
    k = fq.BufferedHead(np.zeros((0, 4), np.float32))
    v = fq.BufferedHead(np.zeros((0, 4), np.float32))
    k.append(np.array([127.0, 0.0, -127.0, 64.0], np.float32))         # u = 1 -> exact
    v.append(np.array([-127.0, 2.0, 0.0, 100.0], np.float32))
    q = np.array([[0.5, 1.0, 0.25, -0.125], [1.0, 0.0, 0.0, 0.0]])
    o, lse = fq.attention_buffered(q, k, v, 0.5)
    assert np.array_equal(o, np.tile([-127.0, 2.0, 0.0, 100.0], (2, 1)))
    assert np.allclose(lse, 0.5 * (q @ np.array([127.0, 0.0, -127.0, 64.0])), rtol=0, atol=1e-12)


def test_dequantize_int8_hand_values():
    got = fq.dequantize_int8(np.array([[3, -2, 127, 0]], np.int8), np.array([0.5], np.float16))
    assert got.tolist() == [[1.5, -1.0, 63.5, 0.0]]


MUTATIONS = [
    ("universal_scale", "r32 / np.float32(QMAX8)", "r32 / np.float32(128)"),          # wrong divisor
    ("quantize_int8", "np.rint(", "np.floor(0.5 + "),                                # ties away from even
    ("quantize_int8", "np.clip(q, -QMAX8, QMAX8)", "np.clip(q, -QMAX8 - 1, QMAX8)"),  # asymmetric clamp
    ("history_range", "np.float32(codec.QMAX) * s.max", "np.float32(8) * s.max"),    # R = 7 x max s
    ("BufferedHead.append", "if self.r == 0:", "if False:"),                         # empty history keeps R = 0
    ("BufferedHead.flush", "max(float(self.r), float(history_range(s)))", "float(history_range(s))"),  # R not kept
    ("dequantize_int8", "np.asarray(c, dtype=np.float64) *", "np.asarray(c, dtype=np.float64) + 0 *"),  # u dropped
]
PINS = [test_universal_scale_closed_forms, test_int8_codes_equal_exact_rounding_and_clamp,
        test_history_range_is_seven_times_the_largest_scale, test_first_row_sets_the_range_of_an_empty_history,
        test_outlier_past_the_range_is_clamped, test_flush_reproduces_representable_rows,
        test_attention_over_one_buffered_key_is_its_value, test_dequantize_int8_hand_values]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] + ":" + m[2] for m in MUTATIONS])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    func, old, new = mutation
    assert mutant_fails_a_pin(monkeypatch, fq, func, old, new, PINS), mutation
