"""Pins of oracle/progressive.py (TurboAttention §3.1: progressive INT8 ->
INT4 storage, channel-wise asymmetric) against hand-derived vectors, exact
rational rounding and closed-form bounds."""

import os
from fractions import Fraction

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import flashq
from oracle import progressive as pq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "progressive_stage2_vectors.txt")


def _vectors():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        q1, sz, q2, back, _ = [x.strip() for x in line.split("|", 4)]
        s2, z2 = (int(v) for v in sz.split())
        out.append(([int(v) for v in q1.split()], s2, z2, [int(v) for v in q2.split()], [int(v) for v in back.split()]))
    return out


@pytest.mark.parametrize("q1,s2,z2,q2,back", _vectors())
def test_stage2_hand_vectors(q1, s2, z2, q2, back):
    c = np.array(q1, dtype=np.int8)[:, None]
    got_q2, got_s2, got_z2 = pq.stage2(c)
    assert int(got_s2[0]) == s2 and int(got_z2[0]) == z2
    assert got_q2[:, 0].tolist() == q2
    assert pq.read_int8(got_q2, got_s2, got_z2)[:, 0].tolist() == back


def test_stage2_rounding_is_round_half_even_on_exact_rationals():
    """Every offset 0..254 against every scale 1..17: Python's round() of an
    exact Fraction (banker's rounding) is the reference."""
    for s2 in range(1, 18):
        hi = min(254, 15 * s2)
        col = np.array([-127] + [-127 + n for n in range(hi + 1)], dtype=np.int64)
        # force the scale: the column's range is exactly hi, so s2 = max(1, ceil(hi / 15))
        q2, got_s2, _ = pq.stage2(np.clip(col, -127, 127).astype(np.int8)[:, None])
        want_s2 = max(1, -(-hi // 15))
        assert int(got_s2[0]) == want_s2
        for n in range(hi + 1):
            assert int(q2[n + 1, 0]) == round(Fraction(n, want_s2)), (s2, n)


def test_stage2_invariants_on_random_blocks():
    rng = np.random.default_rng(0)
    for _ in range(200):
        span = int(rng.integers(0, 255))
        lo = int(rng.integers(-127, 128 - span))
        q1 = rng.integers(lo, lo + span + 1, (64, 8)).astype(np.int8)
        q2, s2, z2 = pq.stage2(q1)
        assert q2.max() <= 15 and (q2.min(axis=0) == 0).all()          # the minimum maps to 0
        rng_c = q1.astype(np.int64).max(axis=0) - q1.astype(np.int64).min(axis=0)
        assert (s2.astype(np.int64) == np.maximum(1, -(-rng_c // 15))).all()
        assert ((s2 == 1) | ((s2.astype(np.int64) - 1) * 15 < rng_c)).all()   # the smallest such integer
        back = pq.read_int8(q2, s2, z2)
        assert (2 * np.abs(back - q1.astype(np.int64)) <= s2.astype(np.int64)).all()   # within s2 / 2
        lossless = rng_c <= 15
        assert (back[:, lossless] == q1[:, lossless]).all()


def test_pack_order_and_round_trip():
    assert pq.pack_unsigned(np.array([1, 2, 15, 0], dtype=np.uint8)).tolist() == [0x21, 0x0F]
    q = np.random.default_rng(1).integers(0, 16, (7, 32)).astype(np.uint8)
    assert np.array_equal(pq.unpack_unsigned(pq.pack_unsigned(q)), q)


def test_stage1_is_the_buffer_code_over_the_block_range():
    """The block's largest magnitude gets code +-127 (scale not saturated);
    codes are the decode buffer's int8 rule with u from the block absmax."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 16)).astype(np.float32)
    q1, s1 = pq.stage1(x)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(int(q1[i])) == 127
    u = flashq.universal_scale(np.max(np.abs(x)))
    assert s1 == u
    assert np.array_equal(q1, flashq.quantize_int8(x, np.full(64, u)))
    zero_q1, zero_s1 = pq.stage1(np.zeros((64, 4), np.float32))
    assert zero_s1 == 0 and not zero_q1.any()


def test_blocks_round_trip_within_the_two_stage_bound():
    """|x^ - x| <= s1 / 2 (stage 1) + s2 * s1 / 2 (stage 2), per element."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3, 128, 32)).astype(np.float32)
    x[0, 1, :, 5] *= 10.0                                    # an outlier channel
    packed, s1, s2, z2 = pq.quantize_blocks(x)
    assert packed.shape == (2, 3, 128, 16) and s1.shape == (2, 3, 2) and s2.shape == (2, 3, 2, 32)
    xh = pq.dequantize_blocks(packed, s1, s2, z2)
    s1b = np.repeat(s1.astype(np.float64), 64, axis=-1)[..., None]
    s2b = np.repeat(s2.astype(np.float64), 64, axis=-2)
    assert (np.abs(xh - x) <= s1b / 2 + s2b * s1b / 2 + 1e-12).all()


def test_compressing_a_full_buffer_uses_its_codes_and_scale():
    rng = np.random.default_rng(4)
    q1 = rng.integers(-127, 128, (64, 8)).astype(np.int8)
    packed, s1, s2, z2 = pq.compress_int8_block(q1, np.float16(0.125))
    q2 = pq.unpack_unsigned(packed)
    xh = pq.dequantize_blocks(packed[None], np.array([s1]), s2[None], z2[None])
    assert np.array_equal(xh[0], pq.read_int8(q2, s2, z2) * 0.125)


def test_constant_channels_store_only_the_zero_point():
    x = np.tile(np.linspace(-1, 1, 8, dtype=np.float32), (64, 1))   # every token equal
    packed, s1, s2, z2 = pq.quantize_blocks(x)
    assert not pq.unpack_unsigned(packed).any() and (s2 == 1).all()
    q1, s = pq.stage1(x)
    assert np.array_equal(z2[0], q1[0]) and s1[0] == s


def _all_hand_vectors():
    for args in _vectors():
        test_stage2_hand_vectors(*args)


MUTATIONS = [
    ("stage1", "np.max(np.abs(x32))", "np.max(x32)"),                            # range without the sign
    ("stage2", "-((lo - hi) // QMAX4)", "(hi - lo) // QMAX4"),                    # floor, not ceiling
    ("stage2", "np.maximum(1, ", "np.maximum(2, "),                               # scale floor off by one
    ("stage2", "(fl % 2 == 1)", "(fl % 2 == 0)"),                                 # ties to odd
    ("stage2", "num = q - lo", "num = q - lo - 1"),                               # zero point off by one
    ("pack_unsigned", "(q[..., 0::2] | (q[..., 1::2] << 4))", "(q[..., 1::2] | (q[..., 0::2] << 4))"),  # nibble order
    ("read_int8", "+ np.asarray(z2", "- np.asarray(z2"),                          # zero point sign
    ("dequantize_blocks", "x = q1.astype(np.float64) *", "x = qb.astype(np.float64) *"),  # nibbles read as int8
    ("compress_int8_block", "np.float16(s1)", "np.float16(1.0)"),                  # buffer scale dropped
]
PINS = [_all_hand_vectors, test_stage2_rounding_is_round_half_even_on_exact_rationals,
        test_stage2_invariants_on_random_blocks, test_pack_order_and_round_trip,
        test_stage1_is_the_buffer_code_over_the_block_range, test_blocks_round_trip_within_the_two_stage_bound,
        test_compressing_a_full_buffer_uses_its_codes_and_scale, test_constant_channels_store_only_the_zero_point]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] + ":" + m[2] for m in MUTATIONS])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    func, old, new = mutation
    assert mutant_fails_a_pin(monkeypatch, pq, func, old, new, PINS), mutation
