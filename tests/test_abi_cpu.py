"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before any launch."""

import ctypes
import subprocess

import pytest

from common import ensure_library, header_symbols

qa = ensure_library()
lib = qa.load_library()


def test_exports_every_declared_symbol():
    declared = header_symbols()
    assert len(declared) >= 9
    nm = subprocess.run(["nm", "-D", "--defined-only", qa.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in nm.splitlines() if line.strip()}
    for name in declared:
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(qa.EXPORTS) == set(declared)


def test_status_strings_and_version():
    assert lib.qattn_version() == 0x000100
    for st in range(5):
        assert lib.qattn_status_string(st)
    assert lib.qattn_status_string(99) == b"unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def _cache(**kw):
    s = qa.KvCacheStruct()
    s.k_codes = s.k_scales = s.v_codes = s.v_scales = FAKE
    s.head_dim, s.num_kv_heads, s.capacity = 128, 2, 256
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def _decode(cache, batch=1, hq=4, max_len=100, splits=0):
    return lib.qattn_decode(FAKE, ctypes.byref(cache), FAKE, batch, hq, max_len, 1.0, splits, None, 0,
                            FAKE, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), qa.QATTN_ERR_UNSUPPORTED),
    (dict(capacity=100), qa.QATTN_ERR_UNSUPPORTED),
    (dict(num_kv_heads=0), qa.QATTN_ERR_INVALID_ARG),
    (dict(k_codes=FAKE + 8), qa.QATTN_ERR_INVALID_ARG),
    (dict(v_scales=0), qa.QATTN_ERR_INVALID_ARG),
    (dict(page_table=FAKE, page_size=32, num_pages=4, max_pages_per_seq=2), qa.QATTN_ERR_UNSUPPORTED),
    (dict(page_table=FAKE, page_size=64, num_pages=0, max_pages_per_seq=2), qa.QATTN_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_cache(kw, status):
    assert _decode(_cache(**kw)) == status
    assert lib.qattn_last_error()


def test_decode_rejects_bad_heads_and_splits():
    assert _decode(_cache(), hq=5) == qa.QATTN_ERR_INVALID_ARG         # Hq % Hkv
    assert _decode(_cache(), hq=18) == qa.QATTN_ERR_UNSUPPORTED        # group 9 > 8
    assert _decode(_cache(), splits=2000) == qa.QATTN_ERR_INVALID_ARG
    assert _decode(_cache(), max_len=-1) == qa.QATTN_ERR_INVALID_ARG
    assert b"multiple" in lib.qattn_last_error() or True
    assert lib.qattn_decode(FAKE, None, FAKE, 1, 4, 10, 1.0, 0, None, 0, FAKE, None, None) == qa.QATTN_ERR_INVALID_ARG


def test_prefill_rejects_bad_arguments():
    c = _cache()
    pf = lambda **kw: lib.qattn_prefill(kw.get("q", FAKE), ctypes.byref(kw.get("cache", c)), 1, kw.get("hq", 4),
                                        kw.get("nq", 10), kw.get("nk", 20), 1.0, kw.get("causal", 1),
                                        kw.get("out", FAKE), None, None)
    assert pf(nq=30, nk=20) == qa.QATTN_ERR_INVALID_ARG                  # nq > nk
    assert pf(nk=300) == qa.QATTN_ERR_INVALID_ARG                        # nk > capacity
    assert pf(causal=2) == qa.QATTN_ERR_INVALID_ARG
    assert pf(q=FAKE + 2) == qa.QATTN_ERR_INVALID_ARG                    # misaligned
    paged = _cache(page_table=FAKE, page_size=64, num_pages=4, max_pages_per_seq=2)  # 128 tokens per sequence
    assert pf(cache=paged, nk=129, nq=10) == qa.QATTN_ERR_INVALID_ARG   # nk beyond the page-table row
    assert pf(cache=_cache(page_table=FAKE, page_size=32, num_pages=4, max_pages_per_seq=2)) == qa.QATTN_ERR_UNSUPPORTED


def test_quantize_and_combine_reject_bad_arguments():
    c = _cache()
    assert lib.qattn_quantize_kv(FAKE, FAKE, 7, 1, 4, None, ctypes.byref(c), None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_quantize_kv(FAKE, FAKE, 0, -1, 4, None, ctypes.byref(c), None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_quantize_kv(None, FAKE, 0, 1, 4, None, ctypes.byref(c), None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_quantize_kv(FAKE, FAKE, 0, 0, 4, None, ctypes.byref(c), None) == qa.QATTN_OK  # nothing to do
    assert lib.qattn_combine(FAKE, FAKE, 0, 4, 128, FAKE, None, None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_combine(FAKE, FAKE, 4, 4, 96, FAKE, None, None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_combine(FAKE, FAKE, 2, 0, 128, FAKE, None, None) == qa.QATTN_OK            # empty


def test_workspace_size_host_arithmetic():
    # Explicit range counts need no device.  A stage carries 256 (token, kv-head)
    # rows: 256 tokens of one kv-head in a contiguous cache, one 64-token page of
    # 4 kv-heads in a paged pool (256/Hkv tokens of all heads when Hkv < 4).  Two
    # partial slots per range, each with (kv-heads per stage * G) rows:
    # partial_o fp32 [2 * ranges, rows, D], then partial_lse [2 * ranges, rows].
    # The query does not know the layout, so it returns the larger need.
    def need(ranges, rows, d):
        return 2 * ranges * rows * d * 4 + 2 * ranges * rows * 4
    # Hkv=2: contiguous ranges min(4, 2*2*ceil(1000/256)) = 4 with G=4 rows;
    # paged stages hold both heads (rows 8), ranges min(4, 2*1*ceil(1000/128)) = 4
    assert qa.decode_workspace_size(2, 8, 2, 128, 1000, 4) == need(4, 8, 128)
    # Hkv=1: 256 tokens per stage either way, ceil(300/256) = 2 ranges, 1 row
    assert qa.decode_workspace_size(1, 1, 1, 64, 300, 9) == need(2, 1, 64)
    assert qa.decode_workspace_size(1, 3, 1, 64, 64, 1) == need(1, 3, 64)
    # Hkv=8, G=4: paged slots hold 4 kv-heads (rows 16)
    assert qa.decode_workspace_size(8, 32, 8, 128, 4096, 152) == need(152, 16, 128)
    # Hkv=6 has no paged geometry (not a multiple of 4): contiguous rows only
    assert qa.decode_workspace_size(2, 12, 6, 128, 600, 4) == need(4, 2, 128)
    assert qa.decode_workspace_size(0, 8, 2, 128, 60, 4) == 0             # invalid sizes
    assert qa.decode_workspace_size(2, 8, 2, 96, 600, 4) == 0
    assert qa.decode_workspace_size(4096, 8, 2, 128, 600, 4) == 0         # batch above the limit


def test_decode_plan_rejects_bad_sizes():
    # invalid sizes are refused on the host, before any device query
    w, n, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    bad = [
        (0, 8, 2, 128, 100, 0, 0, 4, 0),      # no sequence
        (2, 8, 3, 128, 100, 0, 0, 4, 0),      # Hq not a multiple of Hkv
        (2, 8, 2, 96, 100, 0, 0, 4, 0),       # head_dim
        (2, 8, 2, 128, -1, 0, 0, 4, 0),       # negative max length
        (2, 8, 2, 128, 100, 2000, 0, 4, 0),   # too many splits
        (2, 8, 2, 128, 100, 0, 0, 5, 0),      # code bits
        (2, 24, 6, 128, 100, 0, 1, 4, 0),     # paged Hkv = 6
        (2, 72, 2, 128, 100, 0, 0, 4, 0),     # group above QATTN_MAX_GROUP
    ]
    for args in bad:
        assert lib.qattn_decode_plan(*args, ctypes.byref(w), ctypes.byref(n), ctypes.byref(c)) == qa.QATTN_ERR_INVALID_ARG, args


def test_wait_check_rejects_bad_arguments():
    assert lib.qattn_check_wait_timeout(None, 1000, None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_check_wait_timeout(FAKE, 0, None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_check_wait_timeout(FAKE, (1 << 31) + 1, None) == qa.QATTN_ERR_INVALID_ARG


def test_decode_append_rejects_bad_arguments():
    c = _cache()

    def da(k=FAKE, v=FAKE, dt=qa.QATTN_F32, batch=1):
        return lib.qattn_decode_append(FAKE, k, v, dt, ctypes.byref(c), FAKE, batch, 4, 100, 1.0, 0, None, 0,
                                       FAKE, None, None)
    assert da(dt=7) == qa.QATTN_ERR_INVALID_ARG
    assert da(k=None) == qa.QATTN_ERR_INVALID_ARG
    assert da(v=None) == qa.QATTN_ERR_INVALID_ARG
    assert da(k=FAKE + 4) == qa.QATTN_ERR_INVALID_ARG   # misaligned
    assert da(v=FAKE + 8) == qa.QATTN_ERR_INVALID_ARG
    assert da(batch=0) == qa.QATTN_OK                   # nothing to do


def _fq(**kw):
    s = qa.FlashqBufferStruct()
    s.k_codes = s.v_codes = s.k_scale = s.v_scale = s.k_range = s.v_range = s.count = FAKE
    s.head_dim, s.num_kv_heads = 128, 2
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def test_flashq_rejects_bad_arguments():
    c = _cache()
    init = lambda b, cache=c, batch=1: lib.qattn_flashq_init(ctypes.byref(b), ctypes.byref(cache), FAKE, batch, None)
    assert lib.qattn_flashq_init(None, ctypes.byref(c), FAKE, 1, None) == qa.QATTN_ERR_INVALID_ARG
    assert init(_fq(head_dim=96)) == qa.QATTN_ERR_UNSUPPORTED
    assert init(_fq(num_kv_heads=0)) == qa.QATTN_ERR_INVALID_ARG
    assert init(_fq(count=0)) == qa.QATTN_ERR_INVALID_ARG
    assert init(_fq(k_codes=FAKE + 4)) == qa.QATTN_ERR_INVALID_ARG             # misaligned
    assert init(_fq(num_kv_heads=4)) == qa.QATTN_ERR_INVALID_ARG               # cache has Hkv 2
    assert init(_fq(head_dim=64)) == qa.QATTN_ERR_INVALID_ARG                  # cache has D 128
    assert lib.qattn_flashq_init(ctypes.byref(_fq()), ctypes.byref(c), None, 1, None) == qa.QATTN_ERR_INVALID_ARG
    assert init(_fq(), batch=0) == qa.QATTN_OK
    b = _fq()
    assert lib.qattn_flashq_append(FAKE, FAKE, 7, ctypes.byref(b), 1, None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_flashq_append(None, FAKE, 0, ctypes.byref(b), 1, None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_flashq_append(FAKE + 8, FAKE, 0, ctypes.byref(b), 1, None) == qa.QATTN_ERR_INVALID_ARG
    att = lambda hq=4, lse=FAKE, batch=1: lib.qattn_flashq_attend(FAKE, ctypes.byref(b), batch, hq, 1.0, FAKE, lse, None)
    assert att(lse=None) == qa.QATTN_ERR_INVALID_ARG                           # lse is required
    assert att(hq=3) == qa.QATTN_ERR_INVALID_ARG
    assert att(hq=2 * 9) == qa.QATTN_ERR_UNSUPPORTED                           # group of 9
    assert att(batch=0) == qa.QATTN_OK
    assert lib.qattn_flashq_flush(ctypes.byref(_fq(head_dim=64)), ctypes.byref(c), FAKE, 1, None) == qa.QATTN_ERR_INVALID_ARG


def test_int3_cache_checks():
    assert _decode(_cache(code_bits=5)) == qa.QATTN_ERR_INVALID_ARG
    assert _decode(_cache(code_bits=3, head_dim=64)) == qa.QATTN_ERR_UNSUPPORTED
    paged3 = _cache(code_bits=3, page_table=FAKE, page_size=64, num_pages=4, max_pages_per_seq=2)
    assert _decode(paged3) == qa.QATTN_ERR_UNSUPPORTED
    c3 = _cache(code_bits=3)
    assert lib.qattn_prefill(FAKE, ctypes.byref(c3), 1, 4, 8, 8, 1.0, 1, FAKE, None, None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_decode_append(FAKE, FAKE, FAKE, qa.QATTN_F32, ctypes.byref(c3), FAKE, 1, 4, 100, 1.0, 0, None, 0,
                                   FAKE, None, None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_flashq_init(ctypes.byref(_fq()), ctypes.byref(c3), FAKE, 1, None) == qa.QATTN_ERR_UNSUPPORTED


def test_int2_cache_checks():
    assert _decode(_cache(code_bits=1)) == qa.QATTN_ERR_INVALID_ARG
    assert _decode(_cache(code_bits=2, head_dim=64)) == qa.QATTN_ERR_UNSUPPORTED
    paged2 = _cache(code_bits=2, page_table=FAKE, page_size=64, num_pages=4, max_pages_per_seq=2)
    assert _decode(paged2) == qa.QATTN_ERR_UNSUPPORTED
    c2 = _cache(code_bits=2)
    assert lib.qattn_prefill(FAKE, ctypes.byref(c2), 1, 4, 8, 8, 1.0, 1, FAKE, None, None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_decode_append(FAKE, FAKE, FAKE, qa.QATTN_F32, ctypes.byref(c2), FAKE, 1, 4, 100, 1.0, 0, None, 0,
                                   FAKE, None, None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_flashq_init(ctypes.byref(_fq()), ctypes.byref(c2), FAKE, 1, None) == qa.QATTN_ERR_UNSUPPORTED


def test_kv_head_index_checks():
    # a cache holding 2 of a model's 4 kv-heads
    listed = _cache(kv_head_index=FAKE, model_kv_heads=4)
    assert _decode(_cache(kv_head_index=FAKE, model_kv_heads=1)) == qa.QATTN_ERR_INVALID_ARG  # fewer than it holds
    paged = _cache(kv_head_index=FAKE, model_kv_heads=4, page_table=FAKE, page_size=64, num_pages=4,
                   max_pages_per_seq=2)
    assert _decode(paged) == qa.QATTN_ERR_UNSUPPORTED
    assert _decode(listed, hq=6) == qa.QATTN_ERR_INVALID_ARG      # Hq must divide by the model's 4 heads
    assert _decode(listed, hq=4 * 65) == qa.QATTN_ERR_UNSUPPORTED  # group size above the limit
    assert lib.qattn_prefill(FAKE, ctypes.byref(listed), 1, 4, 8, 8, 1.0, 1, FAKE, None, None) == \
        qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_decode_append(FAKE, FAKE, FAKE, qa.QATTN_F32, ctypes.byref(listed), FAKE, 1, 8, 100, 1.0, 0,
                                   None, 0, FAKE, None, None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_flashq_init(ctypes.byref(_fq()), ctypes.byref(listed), FAKE, 1, None) == qa.QATTN_ERR_UNSUPPORTED


def _plan(**kw):
    a = dict(k=FAKE, v=FAKE, dt=qa.QATTN_F32, batch=1, hkv=4, n=16, d=128, lens=None, low=1, bits=FAKE, prio=None)
    a.update(kw)
    return lib.qattn_headwise_plan(a["k"], a["v"], a["dt"], a["batch"], a["hkv"], a["n"], a["d"], a["lens"],
                                   a["low"], a["bits"], a["prio"], None)


def test_headwise_plan_rejects_bad_arguments():
    assert _plan(low=-1) == qa.QATTN_ERR_INVALID_ARG
    assert _plan(low=5) == qa.QATTN_ERR_INVALID_ARG
    assert _plan(hkv=0) == qa.QATTN_ERR_UNSUPPORTED
    assert _plan(hkv=257, low=0) == qa.QATTN_ERR_UNSUPPORTED
    assert _plan(d=96) == qa.QATTN_ERR_UNSUPPORTED
    assert _plan(bits=None) == qa.QATTN_ERR_INVALID_ARG
    assert _plan(k=None) == qa.QATTN_ERR_INVALID_ARG
    assert _plan(dt=7) == qa.QATTN_ERR_INVALID_ARG
    assert _plan(batch=-1) == qa.QATTN_ERR_INVALID_ARG


def test_mixed_caches_split_the_heads_by_width():
    import torch
    bits = torch.tensor([4, 2, 4, 4, 2, 4], dtype=torch.int32)
    c4, c2 = qa.mixed_caches(bits, 3, 100, 128, device="cpu")
    assert c4.kv_head_index.tolist() == [0, 2, 3, 5] and c2.kv_head_index.tolist() == [1, 4]
    assert (c4.code_bits, c2.code_bits) == (4, 2)
    assert c4.model_kv_heads == c2.model_kv_heads == 6
    assert tuple(c4.k_codes.shape) == (3, 4, 128, 64)    # capacity rounded up to whole 64-token stages
    assert tuple(c2.v_codes.shape) == (3, 2, 128, 32)    # INT2: 32 bytes per row at D = 128
    assert c2.workspace_kv_heads == 6
    s = c2.struct()
    assert s.kv_head_index == c2.kv_head_index.data_ptr() and s.model_kv_heads == 6 and s.code_bits == 2
    only4, none2 = qa.mixed_caches([4, 4], 1, 64, 64, device="cpu")
    assert none2 is None and only4.kv_head_index.tolist() == [0, 1]
    plain = qa.KvCache.contiguous(1, 2, 64, 128, device="cpu")
    assert plain.struct().kv_head_index is None and plain.workspace_kv_heads == 2


def test_binding_argument_counts_match_the_header():
    import os
    import re
    from common import ROOT
    with open(os.path.join(ROOT, "include", "qattn.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    decls = re.findall(r"\b(qattn_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S)
    assert len(decls) == len(qa.EXPORTS)
    for name, params in decls:
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(getattr(lib, name).argtypes) == n, name


def test_ctypes_structs_match_the_c_layout(tmp_path):
    """sizeof and every field offset of the two ABI structs, as the C compiler
    lays them out, against the binding's ctypes mirrors."""
    import os
    import shutil
    from common import ROOT
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"qattn_kv_cache": qa.KvCacheStruct, "qattn_flashq_buffer": qa.FlashqBufferStruct,
               "qattn_pq_cache": qa.PqCacheStruct}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "qattn.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("  return 0;\n}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    want = []
    for cname, py in structs.items():
        want.append(f"{cname} size {ctypes.sizeof(py)}")
        want += [f"{cname} {f} {getattr(py, f).offset}" for f, _ in py._fields_]
    assert [l for l in got if l] == want


def test_comparison_and_progressive_calls_reject_bad_arguments():
    """Host checks of the FP16, dequantize and progressive entry points (no GPU work)."""
    qa = ensure_library()
    lib = qa.load_library()
    fake = 0x10000
    st = qa.KvCacheStruct()
    st.k_codes = st.k_scales = st.v_codes = st.v_scales = fake
    st.head_dim, st.num_kv_heads, st.capacity = 128, 8, 4096
    assert lib.qattn_dequantize_kv(ctypes.byref(st), 1, 4097, fake, fake, None) == qa.QATTN_ERR_INVALID_ARG  # n > capacity
    st.code_bits = 3
    assert lib.qattn_dequantize_kv(ctypes.byref(st), 1, 64, fake, fake, None) == qa.QATTN_ERR_UNSUPPORTED
    # fp16 decode: D 96, group 16, capacity 0
    assert lib.qattn_decode_fp16(fake, fake, fake, 1, 8, 8, 96, 64, fake, 64, 1.0, 0, None, 0, fake, None,
                                 None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_decode_fp16(fake, fake, fake, 1, 32, 2, 128, 64, fake, 64, 1.0, 0, None, 0, fake, None,
                                 None) == qa.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_decode_fp16(fake, fake, fake, 1, 8, 8, 128, 0, fake, 64, 1.0, 0, None, 0, fake, None,
                                 None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_decode_fp16_workspace_size(1, 8, 3, 128, 64, 0) == 0                    # Hq % Hkv
    # fp16 prefill: nq > nk, nk > capacity
    assert lib.qattn_prefill_fp16(fake, fake, fake, 1, 8, 8, 128, 256, 100, 50, 1.0, 1, fake, None,
                                  None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_prefill_fp16(fake, fake, fake, 1, 8, 8, 128, 64, 10, 100, 1.0, 1, fake, None,
                                  None) == qa.QATTN_ERR_INVALID_ARG
    # progressive: n not a multiple of 64, capacity not a multiple of 64, NULL pointer
    pq = qa.PqCacheStruct(fake, fake, fake, fake, 128, 8, 4096)
    assert lib.qattn_pq_quantize(fake, fake, 0, 1, 100, None, ctypes.byref(pq), None) == qa.QATTN_ERR_INVALID_ARG
    bad = qa.PqCacheStruct(fake, fake, fake, fake, 128, 8, 100)
    assert lib.qattn_pq_quantize(fake, fake, 0, 1, 64, None, ctypes.byref(bad), None) == qa.QATTN_ERR_INVALID_ARG
    null = qa.PqCacheStruct(0, fake, fake, fake, 128, 8, 4096)
    assert lib.qattn_decode_pq(fake, ctypes.byref(null), fake, 1, 8, 64, 1.0, 0, None, 0, fake, None,
                               None) == qa.QATTN_ERR_INVALID_ARG
    assert lib.qattn_decode_pq(fake, ctypes.byref(pq), fake, 1, 12, 64, 1.0, 0, None, 0, fake, None,
                               None) == qa.QATTN_ERR_INVALID_ARG                              # Hq % Hkv
