"""Pins for the codec oracle (CPU only).

Nothing here retypes the oracle's formula: the expected values come from
hand-derived vectors (tests/golden/codec_vectors.txt), from the byte counts
page 1 prints for a tile (tests/golden/page_figures.txt), from an
exact-rational reimplementation of IEEE rounding, and from invariants the
symmetric codec must satisfy.
"""

import math
import os
from fractions import Fraction as F

import functools

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import codec


# ---------------------------------------------------------------------------
# an independent exact-rational model of the rules
# ---------------------------------------------------------------------------

def _round_binary(fr: F, p: int, emin: int, emax: int):
    """Round a rational to the nearest binary float with a p-bit significand
    (round half to even); returns a Fraction, or None on overflow to inf."""
    if fr == 0:
        return F(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    while F(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)                          # subnormals share emin's ulp
    ulp = F(2) ** (e - (p - 1))
    n = a / ulp
    r = round(n)                              # Fraction.__round__: half to even
    val = r * ulp
    if val >= F(2) ** (emax + 1):
        return None
    return sign * val


def _fl32(fr):
    return _round_binary(fr, 24, -126, 127)


def _fl16_sat(fr):
    v = _round_binary(fr, 11, -14, 15)
    return F(65504) if v is None else v


def exact_row(xs):
    """(scale as Fraction, codes) for one row by exact rational arithmetic."""
    xs = [F(float(v)) for v in xs]
    am = max(abs(v) for v in xs)
    s = _fl16_sat(_fl32(am / 7))
    if s == 0:
        return s, [0] * len(xs)
    codes = [max(-7, min(7, round(v / s))) for v in xs]
    return s, codes


# ---------------------------------------------------------------------------

def _load_vectors(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "codec_vectors.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            xs, sbits, codes, packed, _why = [p.strip() for p in line.split("|")]
            rows.append((
                np.array([float.fromhex(v) for v in xs.split()], dtype=np.float32),
                int(sbits, 16),
                [int(c) for c in codes.split()],
                [int(b, 16) for b in packed.split()],
            ))
    return rows


def test_golden_vectors(golden_dir):
    rows = _load_vectors(golden_dir)
    assert len(rows) >= 10
    for x, sbits, codes, packed in rows:
        c, s = codec.quantize_rows(x[None])
        p, s2 = codec.quantize_pack(x[None])
        assert int(s.view(np.uint16)[0]) == sbits, (x, hex(int(s.view(np.uint16)[0])))
        assert c[0].tolist() == codes, (x, c[0].tolist())
        assert p[0].tolist() == packed, (x, [hex(v) for v in p[0]])
        assert s2.view(np.uint16)[0] == sbits


def test_golden_vectors_match_exact_model(golden_dir):
    # the fixture itself agrees with the exact-rational model of the rules
    for x, sbits, codes, _ in _load_vectors(golden_dir):
        s, cs = exact_row(x)
        assert F(float(np.uint16(sbits).view(np.float16))) == s
        assert cs == codes


def test_page_tile_figures(golden_dir):
    figs = {}
    with open(os.path.join(golden_dir, "page_figures.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                figs[k] = int(v)
    t, d = figs["tile_tokens"], figs["tile_dim"]
    assert codec.tile_bytes(t, d) == (figs["code_bytes"], figs["scale_bytes"])
    x = np.random.default_rng(0).standard_normal((t, d)).astype(np.float32)
    p, s = codec.quantize_pack(x)
    assert p.nbytes == figs["code_bytes"]
    assert s.nbytes == figs["scale_bytes"]


def _rows_with_ties(rng, n, d):
    """Rows whose scale is exact (am = 7 s) with entries at exact half-integers of s."""
    out = []
    for _ in range(n):
        e = int(rng.integers(-10, 10))
        mant = int(rng.integers(1024, 2048))
        s = mant * 2.0 ** (e - 10)                      # an fp16 normal value
        k = rng.integers(-7, 7, size=d).astype(np.float64) + 0.5 * rng.integers(0, 2, size=d)
        row = (k * s).astype(np.float32)
        row[int(rng.integers(0, d))] = np.float32(7 * s) * (1 if rng.random() < .5 else -1)
        out.append(row)
    return np.stack(out)


def test_exact_rational_reference():
    rng = np.random.default_rng(1234)
    d = 8
    blocks = [
        rng.standard_normal((400, d)).astype(np.float32),
        (rng.standard_normal((200, d)) * 10.0 ** rng.uniform(-6, 5, (200, 1))).astype(np.float32),
        _rows_with_ties(rng, 300, d),
        (rng.integers(-15, 16, (200, d)) * 0.5).astype(np.float32),
        (rng.standard_normal((50, d)) * 1e-7).astype(np.float32),   # fp16-subnormal scales
        (rng.standard_normal((20, d)) * 1e6).astype(np.float32),    # saturating scales
    ]
    x = np.concatenate(blocks)
    codes, scales = codec.quantize_rows(x)
    for i in range(x.shape[0]):
        s, cs = exact_row(x[i])
        assert F(float(scales[i])) == s, (x[i], float(scales[i]), float(s))
        assert codes[i].tolist() == cs, (x[i], codes[i].tolist(), cs)


def test_all_fp16_values_against_fixed_absmax():
    # every finite fp16 value v with |v| <= am, in the row [am, v]
    for am in (1.0, 7.0, 3.3, 1000.0, 0.01):
        v = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
        v = np.concatenate([v, -v])
        v = v[np.abs(v) <= np.float32(am)]
        x = np.stack([np.full_like(v, np.float32(am)), v], axis=1)
        codes, scales = codec.quantize_rows(x)
        s = F(float(scales[0]))
        assert (scales == scales[0]).all()
        assert s == exact_row([am, 0.0])[0]
        exact = np.array([max(-7, min(7, round(F(float(t)) / s))) for t in v])
        assert (codes[:, 1] == exact).all()
        assert (codes[:, 0] == 7).all()


def test_invariants():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5000, 128)).astype(np.float32)
    x[:, :4] *= 10.0
    codes, s = codec.quantize_rows(x)
    assert codes.min() >= -7 and codes.max() <= 7
    assert (np.abs(codes).max(axis=1) == 7).all()          # absmax maps to +-7
    s64 = s.astype(np.float64)[:, None]
    err = np.abs(x.astype(np.float64) - codes * s64)
    assert (err <= s64 / 2 * (1 + 1e-12)).all()             # per-element error <= s/2
    # idempotence: the dequantized row re-quantizes to the same codes and scale
    xh = (codes.astype(np.float64) * s64).astype(np.float32)
    codes2, s2 = codec.quantize_rows(xh)
    assert (codes2 == codes).all() and (s2.view(np.uint16) == s.view(np.uint16)).all()


def test_zero_and_tiny_rows():
    x = np.zeros((3, 16), np.float32)
    x[1, 3] = 1e-9                      # scale underflows to 0 -> all codes 0
    x[2, 5] = -np.float32(7 * 2.0 ** -24)  # smallest subnormal scale
    codes, s = codec.quantize_rows(x)
    assert (codes[0] == 0).all() and float(s[0]) == 0.0
    assert (codes[1] == 0).all() and float(s[1]) == 0.0
    assert float(s[2]) == 2.0 ** -24 and codes[2, 5] == -7


def test_pack_layout_and_roundtrip():
    a, b = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    codes = np.stack([a.ravel(), b.ravel()], axis=1).astype(np.int8)
    packed = codec.pack_nibbles(codes)[:, 0]
    for (ca, cb), byte in zip(codes.tolist(), packed.tolist()):
        assert byte == ((ca + 16) % 16) | (((cb + 16) % 16) << 4)
    assert (codec.unpack_nibbles(packed[:, None]) == codes).all()
    allbytes = np.arange(256, dtype=np.uint8)[:, None]
    assert (codec.pack_nibbles(codec.unpack_nibbles(allbytes)) == allbytes).all()


def test_fp16_input_widening():
    rng = np.random.default_rng(3)
    x16 = rng.standard_normal((100, 64)).astype(np.float16)
    p16, s16 = codec.quantize_pack(x16)
    p32, s32 = codec.quantize_pack(x16.astype(np.float32))
    assert (p16 == p32).all() and (s16.view(np.uint16) == s32.view(np.uint16)).all()


def test_dequantize_exact():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 32)).astype(np.float32)
    p, s = codec.quantize_pack(x)
    xh = codec.dequantize(p, s)
    c = codec.unpack_nibbles(p)
    for i in range(4):
        for j in range(32):
            assert F(float(xh[i, j])) == F(int(c[i, j])) * F(float(s[i]))
    # the product is exact in binary32 as well
    assert (xh.astype(np.float32).astype(np.float64) == xh).all()


@pytest.mark.parametrize("mutation", ["half_up", "qmax8", "no_saturation"])
def test_planted_codec_mistakes_are_caught(monkeypatch, golden_dir, mutation):
    """A plausible mistake planted in the oracle must fail a pin."""
    if mutation == "half_up":
        monkeypatch.setattr(codec.np, "rint", lambda q: np.floor(q + 0.5), raising=True)
    elif mutation == "qmax8":
        monkeypatch.setattr(codec, "QMAX", 8)
    elif mutation == "no_saturation":
        monkeypatch.setattr(codec, "FP16_MAX", float("inf"))
    try:
        with pytest.raises(AssertionError):
            test_golden_vectors(golden_dir)
    finally:
        monkeypatch.undo()


SOURCE_MUTATIONS = [
    ("row_scales", "np.max(np.abs(x32), axis=-1)", "np.max(x32, axis=-1)"),                # range without the sign
    ("row_scales", "np.where(np.isinf(s16), np.float16(FP16_MAX), s16)", "np.where(np.isinf(s16), np.float16(0), s16)"),  # overflow to 0
    ("quantize_rows", "np.clip(np.rint(q), -QMAX, QMAX)", "np.clip(np.rint(q), -QMAX - 1, QMAX)"),  # asymmetric clamp
    ("quantize_rows", "q = np.where(s64 > 0.0, x64 / safe, 0.0)", "q = np.where(s64 > 0.0, x64 / safe * 0.999999, 0.0)"),
    ("pack_nibbles", "(lo | (hi << np.uint8(4)))", "(hi | (lo << np.uint8(4)))"),          # nibble order
    ("unpack_nibbles", "lo = np.where(lo >= 8, lo - 16, lo)", "lo = np.where(lo > 8, lo - 16, lo)"),  # -8 read as +8
    ("unpack_nibbles", "hi = np.where(hi >= 8, hi - 16, hi)", "hi = np.where(hi >= 8, hi - 15, hi)"),  # sign extension
    ("dequantize", "return c * np.asarray", "return c * 0.5 * np.asarray"),                 # scale off by two
]


@pytest.mark.parametrize("mutation", SOURCE_MUTATIONS, ids=[m[0] + ":" + m[2][:40] for m in SOURCE_MUTATIONS])
def test_planted_source_mistakes_are_caught(monkeypatch, golden_dir, mutation):
    func, old, new = mutation
    pins = [functools.partial(test_golden_vectors, golden_dir), functools.partial(test_golden_vectors_match_exact_model, golden_dir),
            test_exact_rational_reference, test_all_fp16_values_against_fixed_absmax, test_invariants,
            test_zero_and_tiny_rows, test_pack_layout_and_roundtrip, test_dequantize_exact]
    assert mutant_fails_a_pin(monkeypatch, codec, func, old, new, pins), mutation
