"""Pins for the attention oracle (CPU only).

The oracle is checked against an mpmath brute force (50 digits, plain loops),
against PyTorch's scaled_dot_product_attention in float64 (the textbook
routine for the special case without quantization), against closed forms
(constant V, identical keys, a single key, V = identity), and against the
structural identities the method must satisfy (GQA = repeated MHA, prefill
row = decode prefix, split + combine = unsplit, paged = contiguous).
"""

import inspect
import zlib
import math

import numpy as np
import pytest

from common import mutant_fails_a_pin
from oracle import attention as att
from oracle import codec

mpmath = pytest.importorskip("mpmath")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def brute_force(q, k, v, scale, causal, k_lens=None):
    """Loop-based attention at 50 significant digits."""
    mpmath.mp.dps = 50
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, Hq, Nq, v.shape[-1]))
    L = np.full((B, Hq, Nq), -np.inf)
    for b in range(B):
        nk = Nk if k_lens is None else int(k_lens[b])
        for h in range(Hq):
            kv = h // G
            for i in range(Nq):
                vis = [j for j in range(nk) if (not causal) or j <= i + nk - Nq]
                if not vis:
                    continue
                s = {}
                for j in vis:
                    acc = mpmath.mpf(0)
                    for d in range(D):
                        acc += mpmath.mpf(float(q[b, h, i, d])) * mpmath.mpf(float(k[b, kv, j, d]))
                    s[j] = acc * mpmath.mpf(scale)
                z = mpmath.fsum(mpmath.exp(s[j]) for j in vis)
                for d in range(v.shape[-1]):
                    O[b, h, i, d] = float(mpmath.fsum(mpmath.exp(s[j]) * mpmath.mpf(float(v[b, kv, j, d]))
                                                      for j in vis) / z)
                L[b, h, i] = float(mpmath.log(z))
    return O, L


CASES = [
    # B, Hq, Hkv, Nq, Nk, D, causal, lens
    (1, 1, 1, 1, 1, 4, False, None),
    (1, 2, 1, 3, 5, 4, True, None),
    (2, 4, 2, 4, 4, 8, True, None),
    (2, 4, 2, 1, 7, 6, False, [7, 3]),
    (1, 3, 3, 5, 8, 2, True, None),
    (2, 2, 1, 2, 6, 4, True, [6, 2]),
]


@pytest.mark.parametrize("case", CASES)
def test_brute_force(case):
    B, Hq, Hkv, Nq, Nk, D, causal, lens = case
    rng = np.random.default_rng(zlib.crc32(repr(case).encode()))
    q = _rand(rng, B, Hq, Nq, D).astype(np.float16)
    k = _rand(rng, B, Hkv, Nk, D) * 2
    v = _rand(rng, B, Hkv, Nk, D)
    scale = 1 / math.sqrt(D)
    O, L = att.attention(q, k, v, scale, causal, lens)
    Ob, Lb = brute_force(q, k, v, scale, causal, lens)
    assert np.allclose(O, Ob, atol=1e-12, rtol=0)
    fin = np.isfinite(Lb)
    assert (np.isfinite(L) == fin).all()
    assert np.allclose(L[fin], Lb[fin], atol=1e-12, rtol=0)
    assert (O[~fin] == 0).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq_nk", [(16, 16), (5, 16), (1, 9)])
def test_matches_torch_sdpa_float64(causal, nq_nk):
    torch = pytest.importorskip("torch")
    Nq, Nk = nq_nk
    B, Hq, Hkv, D = 2, 8, 2, 16
    rng = np.random.default_rng(11)
    q = _rand(rng, B, Hq, Nq, D)
    k = _rand(rng, B, Hkv, Nk, D)
    v = _rand(rng, B, Hkv, Nk, D)
    scale = 0.37
    O, _ = att.attention(q, k, v, scale, causal)
    G = Hq // Hkv
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(k).repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).repeat_interleave(G, dim=1)
    mask = None
    if causal:   # bottom-right alignment, written as an explicit boolean mask
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        mask = j <= i + (Nk - Nq)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    assert np.allclose(O, ref.numpy(), atol=1e-12, rtol=0)


def test_closed_forms():
    rng = np.random.default_rng(2)
    B, Hq, Hkv, Nq, Nk, D = 2, 4, 2, 6, 9, 8
    q = _rand(rng, B, Hq, Nq, D)
    k = _rand(rng, B, Hkv, Nk, D)
    # constant V -> O equals that constant
    vconst = np.broadcast_to(rng.standard_normal(D), (B, Hkv, Nk, D))
    O, _ = att.attention(q, k, vconst, 0.5, True)
    assert np.allclose(O, vconst[:, :1, :1].repeat(Hq, 1).repeat(Nq, 2), atol=1e-13)
    # identical keys -> O is the mean of the visible values; lse = s + ln(count)
    v = _rand(rng, B, Hkv, Nk, D)
    krow = rng.standard_normal(D)
    ksame = np.broadcast_to(krow, (B, Hkv, Nk, D))
    O, L = att.attention(q, ksame, v, 0.5, True)
    for b in range(B):
        for h in range(Hq):
            for i in range(Nq):
                n = i + Nk - Nq + 1
                assert np.allclose(O[b, h, i], v[b, h // 2, :n].mean(0), atol=1e-13)
                assert math.isclose(L[b, h, i], 0.5 * q[b, h, i] @ krow + math.log(n), abs_tol=1e-12)
    # a single key -> O = v0 and lse = score
    O, L = att.attention(q, k[:, :, :1], v[:, :, :1], 0.5, False)
    assert np.allclose(O, np.repeat(v[:, :, :1], 2, axis=1).repeat(Nq, 2), atol=1e-14)
    assert np.allclose(L, 0.5 * np.einsum("bhid,bhd->bhi", q, np.repeat(k[:, :, 0], 2, axis=1)), atol=1e-13)


def test_softmax_rows_sum_to_one():
    # with V = identity the output row is the probability row itself
    rng = np.random.default_rng(4)
    Nq, Nk = 7, 12
    q = _rand(rng, 1, 2, Nq, 5)
    k = _rand(rng, 1, 1, Nk, 5) * 3
    v = np.eye(Nk)[None, None]
    for causal in (False, True):
        P, _ = att.attention(q, k, v, 1.0, causal)
        assert (P >= 0).all()
        assert np.allclose(P.sum(-1), 1.0, atol=1e-14)
        if causal:
            i = np.arange(Nq)[:, None]
            j = np.arange(Nk)[None, :]
            assert (P[0, :, j > i + Nk - Nq] == 0).all()


def test_gqa_equals_repeated_mha():
    rng = np.random.default_rng(6)
    q = _rand(rng, 2, 8, 4, 8)
    k = _rand(rng, 2, 2, 10, 8)
    v = _rand(rng, 2, 2, 10, 8)
    O1, L1 = att.attention(q, k, v, 0.3, True)
    O2, L2 = att.attention(q, np.repeat(k, 4, 1), np.repeat(v, 4, 1), 0.3, True)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_prefill_row_equals_decode_prefix():
    rng = np.random.default_rng(8)
    N, D = 11, 8
    q = _rand(rng, 1, 4, N, D)
    k = _rand(rng, 1, 2, N, D)
    v = _rand(rng, 1, 2, N, D)
    O, L = att.attention(q, k, v, 0.4, True)
    for i in range(N):
        Od, Ld = att.attention(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], 0.4, False)
        assert np.allclose(O[:, :, i], Od[:, :, 0], atol=1e-14)
        assert np.allclose(L[:, :, i], Ld[:, :, 0], atol=1e-14)
    # chunked prefill: the last Nq rows of a causal square equal Nq < Nk
    Oc, Lc = att.attention(q[:, :, 7:], k, v, 0.4, True)
    assert np.allclose(Oc, O[:, :, 7:], atol=1e-14) and np.allclose(Lc, L[:, :, 7:], atol=1e-14)


@pytest.mark.parametrize("bounds", [[0, 5, 9, 16], [0, 16], [0, 0, 3, 16, 20], [0, 1, 2, 3, 16]])
def test_split_combine_equals_unsplit(bounds):
    rng = np.random.default_rng(9)
    q = _rand(rng, 2, 4, 1, 8)
    k = _rand(rng, 2, 2, 16, 8)
    v = _rand(rng, 2, 2, 16, 8)
    lens = [16, 7]
    O, L = att.attention(q, k, v, 0.6, False, lens)
    po, pl = att.split_partials(q, k, v, 0.6, bounds, lens)
    Oc, Lc = att.combine(po, pl)
    assert np.allclose(Oc, O, atol=1e-14) and np.allclose(Lc, L, atol=1e-13)


def test_combine_closed_forms():
    # two equal partials merge to the same O and lse + ln 2
    o = np.random.default_rng(1).standard_normal((1, 3, 4))
    l = np.array([[0.5, -1.0, 2.0]])
    O, L = att.combine(np.stack([o[0], o[0]]), np.stack([l[0], l[0]]))
    assert np.allclose(O, o[0]) and np.allclose(L, l[0] + math.log(2))
    # an empty partial carries no weight; all-empty gives O = 0, lse = -inf
    O, L = att.combine(np.stack([o[0], 5 * o[0]]), np.stack([l[0], np.full(3, -np.inf)]))
    assert np.allclose(O, o[0]) and np.allclose(L, l[0])
    O, L = att.combine(np.stack([o[0]]), np.full((1, 3), -np.inf))
    assert (O == 0).all() and np.isneginf(L).all()
    # partial sums of exponentials 1 and 3 (lse 0 and ln 3): weights 1/4 and 3/4, lse ln 4
    a, b = np.array([[1.0, -2.0]]), np.array([[5.0, 2.0]])
    O, L = att.combine(np.stack([a, b]), np.array([[0.0], [math.log(3.0)]]))
    assert np.allclose(O, [[4.0, 1.0]], rtol=0, atol=1e-15) and np.allclose(L, [math.log(4.0)], rtol=0, atol=1e-15)
    # a shift of every lse moves the result's lse by the same amount and leaves O
    O2, L2 = att.combine(np.stack([a, b]), np.array([[700.0], [700.0 + math.log(3.0)]]))
    assert np.allclose(O2, O, rtol=0, atol=1e-13) and np.allclose(L2, L + 700.0, rtol=0, atol=1e-12)


def test_empty_sequence():
    rng = np.random.default_rng(10)
    q = _rand(rng, 2, 2, 1, 4)
    k = _rand(rng, 2, 1, 5, 4)
    O, L = att.attention(q, k, k, 1.0, False, [0, 5])
    assert (O[0] == 0).all() and np.isneginf(L[0]).all()
    assert np.isfinite(L[1]).all()


def _paged_case(rng, lens, Hkv=2, D=8, page=4):
    need = [-(-n // page) for n in lens]
    P = sum(need)
    perm = rng.permutation(P)
    table = -np.ones((len(lens), max(need) + 1), np.int64)
    c = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[c:c + n]
        c += n
    x = rng.standard_normal((P, Hkv, page, D)).astype(np.float32)
    pp, ps = codec.quantize_pack(x)
    return pp, ps, table


def test_paged_equals_contiguous_and_permutation_invariance():
    rng = np.random.default_rng(12)
    lens = [9, 4, 13]
    page = 4
    pk, sk, table = _paged_case(rng, lens, page=page)
    pv, sv, _ = _paged_case(np.random.default_rng(13), lens, page=page)
    pv, sv = pv[: pk.shape[0]], sv[: pk.shape[0]]
    q = rng.standard_normal((3, 4, 1, 8)).astype(np.float16)
    ck, cks = att.gather_pages(pk, sk, table, lens, page)
    cv, cvs = att.gather_pages(pv, sv, table, lens, page)
    O, L = att.attention_quantized(q, ck, cks, cv, cvs, 0.35, False, lens)
    # token t of sequence b is physical (page_table[b, t // page], t % page)
    for b, n in enumerate(lens):
        for t in range(n):
            assert (ck[b, :, t] == pk[table[b, t // page], :, t % page]).all()
    # permuting the pool together with the table leaves the result unchanged
    perm = rng.permutation(pk.shape[0])
    inv = np.argsort(perm)
    table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1)
    ck2, cks2 = att.gather_pages(pk[perm], sk[perm], table2, lens, page)
    cv2, cvs2 = att.gather_pages(pv[perm], sv[perm], table2, lens, page)
    O2, L2 = att.attention_quantized(q, ck2, cks2, cv2, cvs2, 0.35, False, lens)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


def test_gather_pages_literal_example():
    """A hand-written pool and table with the gathered result written out by
    hand (not by the gather formula): pages of 2 tokens, two kv-heads, one code
    byte per token.  Byte value 100 * page + 10 * head + slot; scale value
    page + slot / 4 + head / 8."""
    P, H, page = 3, 2, 2
    pool = np.zeros((P, H, page, 1), dtype=np.uint8)
    sc = np.zeros((P, H, page), dtype=np.float16)
    for p in range(P):
        for h in range(H):
            for o in range(page):
                pool[p, h, o, 0] = 100 * p + 10 * h + o
                sc[p, h, o] = p + o / 4 + h / 8
    table = np.array([[2, 0], [1, -1]])
    lens = [3, 2]
    got_p, got_s = att.gather_pages(pool, sc, table, lens, page)
    # sequence 0: tokens 0, 1 in page 2; token 2 in page 0, slot 0
    # sequence 1: tokens 0, 1 in page 1; its third row is past its length: zero
    want_p = np.array([[[200, 201, 0], [210, 211, 10]],
                       [[100, 101, 0], [110, 111, 0]]], dtype=np.uint8)[..., None]
    want_s = np.array([[[2.0, 2.25, 0.0], [2.125, 2.375, 0.125]],
                       [[1.0, 1.25, 0.0], [1.125, 1.375, 0.0]]], dtype=np.float16)
    assert np.array_equal(got_p, want_p)
    assert np.array_equal(got_s.view(np.uint16), want_s.view(np.uint16))


# ---------------------------------------------------------------------------
# planted mistakes: each one, put into the oracle on the CPU, must fail a pin
# ---------------------------------------------------------------------------

MUTATIONS = [
    ("h // G", "h % Hkv"),                                  # wrong GQA index
    ("j <= i + nk - Nq", "j <= i"),                          # top-left causal
    ("rowmax[live] + np.log(Z)", "np.log(Z)"),               # dropped term in lse
    ("P = E / Z[:, None]", "P = E"),                         # missing normalisation
    ("q[b, h] @ k_hat[b, kv, :nk].T", "q[b, h] @ v_hat[b, kv, :nk].T"),  # wrong operand
    ("softmax_scale * (", "(1.0 + 0 * softmax_scale) * ("),  # dropped scale
]


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_planted_attention_mistakes_are_caught(monkeypatch, mutation):
    src = inspect.getsource(att.attention)
    old, new = mutation
    assert old in src
    ns = dict(vars(att))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(att, "attention", ns["attention"])
    failed = False
    for case in CASES:
        try:
            test_brute_force(case)
        except (AssertionError, ValueError, IndexError):
            failed = True
            break
    assert failed, f"mutation {mutation} was not caught"


GATHER_MUTATIONS = [
    ("page_table[b][t // page_size]", "page_table[b][t % page_size]"),  # page and slot swapped
    ("off = t % page_size", "off = t // page_size"),
    ("out_s[b, :, t] = pool_scales[page, :, off]", "out_s[b, :, t] = pool_scales[page, :, 0]"),
    ("for t in range(seq_lens[b])", "for t in range(L)"),                # rows past the length filled
]


@pytest.mark.parametrize("mutation", GATHER_MUTATIONS)
def test_planted_gather_mistakes_are_caught(monkeypatch, mutation):
    src = inspect.getsource(att.gather_pages)
    old, new = mutation
    assert old in src
    ns = dict(vars(att))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(att, "gather_pages", ns["gather_pages"])
    with pytest.raises((AssertionError, IndexError)):
        test_gather_pages_literal_example()


def _all_split_cases():
    for bounds in ([0, 5, 9, 16], [0, 16], [0, 0, 3, 16, 20], [0, 1, 2, 3, 16]):
        test_split_combine_equals_unsplit(bounds)


COMBINE_MUTATIONS = [
    ("combine", "lse = np.where(live, m_safe + np.log(Zs)", "lse = np.where(live, np.log(Zs)"),  # max dropped from lse
    ("combine", "np.exp(pl - m_safe[None])", "np.exp(pl)"),                                        # unshifted exponentials
    ("combine", "(w[..., None] * po).sum(axis=0) / Zs[..., None]", "(w[..., None] * po).sum(axis=0)"),  # no normalisation
    ("combine", "(w[..., None] * po).sum(axis=0)", "po.sum(axis=0)"),                              # unweighted
    ("split_partials", "sub_lens = [max(0, min(hi, n) - lo) for n in lens]", "sub_lens = [w0 for w0 in [max(hi - lo, 0)] * len(lens)]"),
]


@pytest.mark.parametrize("mutation", COMBINE_MUTATIONS, ids=[m[0] + ":" + m[2][:40] for m in COMBINE_MUTATIONS])
def test_planted_combine_mistakes_are_caught(monkeypatch, mutation):
    func, old, new = mutation
    assert mutant_fails_a_pin(monkeypatch, att, func, old, new, [test_combine_closed_forms, _all_split_cases]), mutation
