"""Python binding of libqattn: INT4-KV attention on GB300 (sm_103a).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  PyTorch provides device memory and the current
stream.  The calls mirror the C ABI in include/qattn.h:

    quantize_kv(k, v, cache, start_pos=None)          quantize-on-append
    decode(q, cache, seq_lens, max_seq_len, scale)    one query per sequence
    decode_plan(batch, Hq, Hkv, D, max_len, splits) the launch shape a decode takes
    prefill(q, cache, nq, nk, scale, causal)          Nq queries per sequence
    combine(partial_o, partial_lse)                   log-sum-exp merge
    dequantize_kv, decode_fp16, prefill_fp16          the comparison paths (FP16 cache;
                                                      dequantize to FP16, then attend)
    pq_quantize, decode_pq                            progressive INT8 -> INT4 blocks

There is no fallback: if libqattn.so is missing or fails to load, every call
raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqattn.so")

QATTN_OK, QATTN_ERR_INVALID_ARG, QATTN_ERR_UNSUPPORTED, QATTN_ERR_WORKSPACE, QATTN_ERR_CUDA = range(5)
QATTN_F32, QATTN_F16 = 0, 1
PAGE_SIZE = 64
MAX_GROUP = 8
MAX_SPLITS = 1024
FLAG_WAIT_TIMEOUT, FLAG_BAD_PAGE, FLAG_TMEM, FLAG_BUFFER_FULL, FLAG_BAD_HEAD = 1, 2, 4, 8, 16
FLASHQ_ROWS = 64

# Every symbol include/qattn.h declares.
EXPORTS = (
    "qattn_quantize_kv", "qattn_decode_workspace_size", "qattn_decode", "qattn_prefill",
    "qattn_combine", "qattn_read_device_flags", "qattn_status_string", "qattn_last_error",
    "qattn_version", "qattn_decode_noalloc", "qattn_check_wait_timeout", "qattn_decode_append",
    "qattn_flashq_init", "qattn_flashq_append", "qattn_flashq_attend", "qattn_flashq_flush",
    "qattn_headwise_plan", "qattn_dequantize_kv", "qattn_decode_fp16_workspace_size", "qattn_decode_fp16",
    "qattn_prefill_fp16", "qattn_pq_quantize", "qattn_decode_pq_workspace_size", "qattn_decode_pq",
    "qattn_flashq_flush_pq", "qattn_decode_plan",
)


class QattnError(RuntimeError):
    """A non-OK status returned by libqattn."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class KvCacheStruct(ctypes.Structure):
    """Layout of ``qattn_kv_cache``."""
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("head_dim", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("max_pages_per_seq", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("capacity", ctypes.c_int64),
        ("num_pages", ctypes.c_int64),
        ("code_bits", ctypes.c_int32),
        ("kv_head_index", ctypes.c_void_p),
        ("model_kv_heads", ctypes.c_int32),
    ]


class PqCacheStruct(ctypes.Structure):
    """Layout of ``qattn_pq_cache``."""
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_params", ctypes.c_void_p),
        ("v_params", ctypes.c_void_p),
        ("head_dim", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("capacity", ctypes.c_int64),
    ]


class FlashqBufferStruct(ctypes.Structure):
    """Layout of ``qattn_flashq_buffer``."""
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("k_range", ctypes.c_void_p),
        ("v_range", ctypes.c_void_p),
        ("count", ctypes.c_void_p),
        ("head_dim", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
    ]


_lib_handle = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqattn.so (once) and declare the C signatures."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run quantized_kv_attention_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    cache_p = ctypes.POINTER(KvCacheStruct)
    sig = {
        "qattn_quantize_kv": (i32, [vp, vp, i32, i32, i32, vp, cache_p, vp]),
        "qattn_decode_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
        "qattn_decode_plan": (i32, [i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp]),
        "qattn_decode": (i32, [vp, cache_p, vp, i32, i32, i32, f32, i32, vp, sz, vp, vp, vp]),
        "qattn_prefill": (i32, [vp, cache_p, i32, i32, i32, i32, f32, i32, vp, vp, vp]),
        "qattn_combine": (i32, [vp, vp, i32, i64, i32, vp, vp, vp]),
        "qattn_read_device_flags": (i32, [ctypes.POINTER(ctypes.c_uint32), i32]),
        "qattn_status_string": (ctypes.c_char_p, [i32]),
        "qattn_last_error": (ctypes.c_char_p, []),
        "qattn_version": (i32, []),
        "qattn_decode_noalloc": (i32, [vp, cache_p, vp, i32, i32, i32, f32, i32, vp, vp, vp]),
        "qattn_check_wait_timeout": (i32, [vp, i64, vp]),
        "qattn_decode_append": (i32, [vp, vp, vp, i32, cache_p, vp, i32, i32, i32, f32, i32, vp, sz, vp, vp, vp]),
        "qattn_flashq_init": (i32, [ctypes.POINTER(FlashqBufferStruct), cache_p, vp, i32, vp]),
        "qattn_flashq_append": (i32, [vp, vp, i32, ctypes.POINTER(FlashqBufferStruct), i32, vp]),
        "qattn_flashq_attend": (i32, [vp, ctypes.POINTER(FlashqBufferStruct), i32, i32, f32, vp, vp, vp]),
        "qattn_flashq_flush": (i32, [ctypes.POINTER(FlashqBufferStruct), cache_p, vp, i32, vp]),
        "qattn_headwise_plan": (i32, [vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp, vp]),
        "qattn_dequantize_kv": (i32, [cache_p, i32, i32, vp, vp, vp]),
        "qattn_decode_fp16_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
        "qattn_decode_fp16": (i32, [vp, vp, vp, i32, i32, i32, i32, i64, vp, i32, f32, i32, vp, sz, vp, vp, vp]),
        "qattn_prefill_fp16": (i32, [vp, vp, vp, i32, i32, i32, i32, i64, i32, i32, f32, i32, vp, vp, vp]),
        "qattn_pq_quantize": (i32, [vp, vp, i32, i32, i32, vp, ctypes.POINTER(PqCacheStruct), vp]),
        "qattn_decode_pq_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
        "qattn_decode_pq": (i32, [vp, ctypes.POINTER(PqCacheStruct), vp, i32, i32, i32, f32, i32, vp, sz, vp, vp, vp]),
        "qattn_flashq_flush_pq": (i32, [ctypes.POINTER(FlashqBufferStruct), ctypes.POINTER(PqCacheStruct), vp, i32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib_handle = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != QATTN_OK:
        lib = load_library()
        msg = lib.qattn_last_error().decode()
        raise QattnError(status, f"{what}: {lib.qattn_status_string(status).decode()}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


@dataclass
class KvCache:
    """Caller-owned INT4 (or INT3, INT2) KV cache (contiguous or paged) as torch tensors.

    contiguous: codes [B, Hkv, capacity, D/2] uint8, scales [B, Hkv, capacity] fp16
    paged:      codes [P, Hkv, 64, D/2] uint8, scales [P, Hkv, 64] fp16,
                page_table [B, max_pages] int32 (-1 = no page)
    code_bits = 3: INT3 rows of 13 little-endian 32-bit words (52 bytes) at D = 128,
                contiguous only (codes [B, Hkv, capacity, 52] uint8)
    code_bits = 2: INT2 rows of 8 words (32 bytes) at D = 128, contiguous only
    kv_head_index: int32 [Hkv] (device): cache head h is the model's kv-head
                kv_head_index[h] of model_kv_heads (headwise mixed precision)
    """
    k_codes: torch.Tensor
    k_scales: torch.Tensor
    v_codes: torch.Tensor
    v_scales: torch.Tensor
    head_dim: int
    num_kv_heads: int
    capacity: int = 0
    page_table: Optional[torch.Tensor] = None
    num_pages: int = 0
    code_bits: int = 4
    kv_head_index: Optional[torch.Tensor] = None
    model_kv_heads: int = 0

    @staticmethod
    def contiguous(batch, num_kv_heads, capacity, head_dim, device="cuda", code_bits=4):
        cap = -(-capacity // PAGE_SIZE) * PAGE_SIZE
        row = 4 * (-(-head_dim // 10)) if code_bits == 3 else head_dim * code_bits // 8
        codes = lambda: torch.zeros(batch, num_kv_heads, cap, row, dtype=torch.uint8, device=device)
        scales = lambda: torch.zeros(batch, num_kv_heads, cap, dtype=torch.float16, device=device)
        return KvCache(codes(), scales(), codes(), scales(), head_dim, num_kv_heads, capacity=cap,
                       code_bits=code_bits)

    @staticmethod
    def paged(num_pages, num_kv_heads, head_dim, page_table, device="cuda"):
        codes = lambda: torch.zeros(num_pages, num_kv_heads, PAGE_SIZE, head_dim // 2, dtype=torch.uint8, device=device)
        scales = lambda: torch.zeros(num_pages, num_kv_heads, PAGE_SIZE, dtype=torch.float16, device=device)
        pt = page_table.to(device=device, dtype=torch.int32).contiguous()
        return KvCache(codes(), scales(), codes(), scales(), head_dim, num_kv_heads,
                       page_table=pt, num_pages=num_pages)

    @property
    def workspace_kv_heads(self) -> int:
        """The kv-head count that sizes a decode workspace (the model's for a listed cache)."""
        return self.model_kv_heads if self.kv_head_index is not None else self.num_kv_heads

    @property
    def paged_layout(self) -> bool:
        return self.page_table is not None

    def struct(self) -> KvCacheStruct:
        s = KvCacheStruct()
        s.k_codes, s.k_scales = self.k_codes.data_ptr(), self.k_scales.data_ptr()
        s.v_codes, s.v_scales = self.v_codes.data_ptr(), self.v_scales.data_ptr()
        s.head_dim, s.num_kv_heads = self.head_dim, self.num_kv_heads
        s.code_bits = self.code_bits
        if self.kv_head_index is not None:
            s.kv_head_index = self.kv_head_index.data_ptr()
            s.model_kv_heads = self.model_kv_heads
        if self.page_table is not None:
            s.page_table = self.page_table.data_ptr()
            s.max_pages_per_seq = self.page_table.shape[1]
            s.page_size = PAGE_SIZE
            s.num_pages = self.num_pages
        else:
            s.page_table = None
            s.capacity = self.capacity
        return s


def quantize_kv(k: torch.Tensor, v: torch.Tensor, cache: KvCache,
                start_pos: Optional[torch.Tensor] = None) -> None:
    """Quantize k, v [B, Hkv, n, D] (fp32 or fp16) into the cache at start_pos[b] + i."""
    if k.dtype not in (torch.float32, torch.float16) or v.dtype != k.dtype:
        raise TypeError("k and v must both be float32 or float16")
    k, v = k.contiguous(), v.contiguous()
    B, _, n, _ = k.shape
    sp = None if start_pos is None else start_pos.to(device=k.device, dtype=torch.int32).contiguous()
    st = cache.struct()
    dt = QATTN_F16 if k.dtype == torch.float16 else QATTN_F32
    _check(load_library().qattn_quantize_kv(_ptr(k), _ptr(v), dt, B, n, _ptr(sp), ctypes.byref(st),
                                            _stream(k.device)), "qattn_quantize_kv")


def decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_splits=0) -> int:
    return int(load_library().qattn_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                          max_seq_len, num_splits))


def decode_plan(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_splits=0, paged=False, code_bits=4,
                listed=False) -> dict:
    """The launch shape of a decode call on the current device: consumer warps
    per CTA, CTAs, and the segment-cluster size (0: cost-balanced ranges and a
    merge kernel)."""
    w, n, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().qattn_decode_plan(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_splits,
                                            int(paged), code_bits, int(listed), ctypes.byref(w), ctypes.byref(n),
                                            ctypes.byref(c)), "qattn_decode_plan")
    return {"warps": w.value, "ctas": n.value, "cluster": c.value}


def decode(q: torch.Tensor, cache: KvCache, seq_lens: torch.Tensor, max_seq_len: int,
           softmax_scale: float, num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
           return_lse: bool = False):
    """q [B, Hq, D] fp16 -> out [B, Hq, D] fp16 (and lse [B, Hq] fp32).  A cache
    with a kv_head_index writes only the rows of the q-heads its kv-heads serve
    (pass `out` / `lse` to collect several such caches; see decode_mixed)."""
    q = q.contiguous()
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if workspace is None:  # a given workspace is checked by the library itself
        need = decode_workspace_size(B, Hq, cache.workspace_kv_heads, D, max_seq_len, num_splits)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    sl = seq_lens.to(device=q.device, dtype=torch.int32).contiguous()
    st = cache.struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().qattn_decode(_ptr(q), ctypes.byref(st), _ptr(sl), B, Hq, max_seq_len,
                                       float(softmax_scale), num_splits, _ptr(workspace), ws_bytes,
                                       _ptr(out), _ptr(lse), _stream(q.device)), "qattn_decode")
    return (out, lse) if return_lse else out


def decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, cache: KvCache,
                  seq_lens: torch.Tensor, max_seq_len: int, softmax_scale: float, num_splits: int = 0,
                  workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None, return_lse: bool = False):
    """One decoding step in one launch: k_new, v_new [B, Hkv, D] (fp32 or fp16)
    are quantized into the cache at position seq_lens[b] - 1 (lengths after the
    append), then q [B, Hq, D] fp16 attends over all seq_lens[b] keys."""
    q = q.contiguous()
    B, Hq, D = q.shape
    if k_new.dtype != v_new.dtype or k_new.dtype not in (torch.float32, torch.float16):
        raise ValueError("k_new and v_new must both be float32 or both float16")
    k_new, v_new = k_new.contiguous(), v_new.contiguous()
    dt = QATTN_F16 if k_new.dtype == torch.float16 else QATTN_F32
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if workspace is None:  # a given workspace is checked by the library itself
        need = decode_workspace_size(B, Hq, cache.workspace_kv_heads, D, max_seq_len, num_splits)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    sl = seq_lens.to(device=q.device, dtype=torch.int32).contiguous()
    st = cache.struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().qattn_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), dt, ctypes.byref(st), _ptr(sl),
                                              B, Hq, max_seq_len, float(softmax_scale), num_splits,
                                              _ptr(workspace), ws_bytes, _ptr(out), _ptr(lse), _stream(q.device)),
           "qattn_decode_append")
    return (out, lse) if return_lse else out


@dataclass
class FlashqBuffer:
    """Caller-owned decode buffer (qattn_flashq_buffer): 64 int8 rows per
    (sequence, kv-head) for K and V, their universal scales and ranges, and the
    number of rows buffered per sequence."""
    k_codes: torch.Tensor   # [B, Hkv, 64, D] int8
    v_codes: torch.Tensor
    k_scale: torch.Tensor   # [B, Hkv] fp16
    v_scale: torch.Tensor
    k_range: torch.Tensor   # [B, Hkv] fp32
    v_range: torch.Tensor
    count: torch.Tensor     # [B] int32
    head_dim: int
    num_kv_heads: int

    @staticmethod
    def create(batch, num_kv_heads, head_dim, device="cuda"):
        codes = lambda: torch.zeros(batch, num_kv_heads, FLASHQ_ROWS, head_dim, dtype=torch.int8, device=device)
        half = lambda: torch.zeros(batch, num_kv_heads, dtype=torch.float16, device=device)
        f32 = lambda: torch.zeros(batch, num_kv_heads, dtype=torch.float32, device=device)
        return FlashqBuffer(codes(), codes(), half(), half(), f32(), f32(),
                            torch.zeros(batch, dtype=torch.int32, device=device), head_dim, num_kv_heads)

    def struct(self) -> FlashqBufferStruct:
        s = FlashqBufferStruct()
        s.k_codes, s.v_codes = self.k_codes.data_ptr(), self.v_codes.data_ptr()
        s.k_scale, s.v_scale = self.k_scale.data_ptr(), self.v_scale.data_ptr()
        s.k_range, s.v_range = self.k_range.data_ptr(), self.v_range.data_ptr()
        s.count = self.count.data_ptr()
        s.head_dim, s.num_kv_heads = self.head_dim, self.num_kv_heads
        return s


def flashq_init(buf: FlashqBuffer, cache: KvCache, cache_lens: torch.Tensor) -> None:
    """Universal scales from the first cache_lens[b] cached rows; empty buffers."""
    cl = cache_lens.to(device=buf.count.device, dtype=torch.int32).contiguous()
    bs, cs = buf.struct(), cache.struct()
    _check(load_library().qattn_flashq_init(ctypes.byref(bs), ctypes.byref(cs), _ptr(cl), cl.numel(),
                                            _stream(buf.count.device)), "qattn_flashq_init")


def flashq_append(k_new: torch.Tensor, v_new: torch.Tensor, buf: FlashqBuffer) -> None:
    """One new K and V row per (sequence, kv-head), [B, Hkv, D] fp32 or fp16."""
    if k_new.dtype != v_new.dtype or k_new.dtype not in (torch.float32, torch.float16):
        raise ValueError("k_new and v_new must both be float32 or both float16")
    k_new, v_new = k_new.contiguous(), v_new.contiguous()
    dt = QATTN_F16 if k_new.dtype == torch.float16 else QATTN_F32
    bs = buf.struct()
    _check(load_library().qattn_flashq_append(_ptr(k_new), _ptr(v_new), dt, ctypes.byref(bs), k_new.shape[0],
                                              _stream(k_new.device)), "qattn_flashq_append")


def flashq_attend(q: torch.Tensor, buf: FlashqBuffer, softmax_scale: float, out: torch.Tensor,
                  lse: torch.Tensor) -> None:
    """Merge attention over the buffered rows into out / lse (a decode over the cached rows)."""
    q = q.contiguous()
    B, Hq, _ = q.shape
    bs = buf.struct()
    _check(load_library().qattn_flashq_attend(_ptr(q), ctypes.byref(bs), B, Hq, float(softmax_scale), _ptr(out),
                                              _ptr(lse), _stream(q.device)), "qattn_flashq_attend")


def flashq_flush(buf: FlashqBuffer, cache: KvCache, cache_lens: torch.Tensor) -> None:
    """Full buffers -> 64 INT4 rows each at positions cache_lens[b] .. + 63."""
    cl = cache_lens.to(device=buf.count.device, dtype=torch.int32).contiguous()
    bs, cs = buf.struct(), cache.struct()
    _check(load_library().qattn_flashq_flush(ctypes.byref(bs), ctypes.byref(cs), _ptr(cl), cl.numel(),
                                             _stream(buf.count.device)), "qattn_flashq_flush")


def prefill(q: torch.Tensor, cache: KvCache, nk: int, softmax_scale: float, causal: bool = True,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            return_lse: bool = False):
    """q [B, Hq, Nq, D] fp16 against the first nk cached keys -> out [B, Hq, Nq, D] fp16."""
    q = q.contiguous()
    B, Hq, Nq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    st = cache.struct()
    _check(load_library().qattn_prefill(_ptr(q), ctypes.byref(st), B, Hq, Nq, nk, float(softmax_scale),
                                        int(bool(causal)), _ptr(out), _ptr(lse), _stream(q.device)),
           "qattn_prefill")
    return (out, lse) if return_lse else out


# ------------------------------------------------------------ comparison paths
# An FP16 KV cache attended directly, and the INT4 cache dequantized to FP16
# in HBM first ("Quantized Cross-Attention ... In-SRAM Dequantization" §5.2):
# the arms the fused kernels are measured against.

def dequantize_kv(cache: KvCache, batch: int, n: int, k_out: Optional[torch.Tensor] = None,
                  v_out: Optional[torch.Tensor] = None):
    """The first n tokens of an INT4 cache as fp16 K, V [batch, Hkv, n, D] (fl16(c * s))."""
    shape = (batch, cache.num_kv_heads, n, cache.head_dim)
    dev = cache.k_codes.device
    k_out = torch.empty(shape, dtype=torch.float16, device=dev) if k_out is None else k_out
    v_out = torch.empty(shape, dtype=torch.float16, device=dev) if v_out is None else v_out
    st = cache.struct()
    _check(load_library().qattn_dequantize_kv(ctypes.byref(st), batch, n, _ptr(k_out), _ptr(v_out), _stream(dev)),
           "qattn_dequantize_kv")
    return k_out, v_out


def decode_fp16_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_splits=0) -> int:
    return int(load_library().qattn_decode_fp16_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                               max_seq_len, num_splits))


def decode_fp16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                softmax_scale: float, num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, return_lse: bool = False):
    """q [B, Hq, D] fp16 against an fp16 cache k, v [B, Hkv, capacity, D] -> out [B, Hq, D] fp16."""
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    B, Hq, D = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if workspace is None:
        need = decode_fp16_workspace_size(B, Hq, Hkv, D, max_seq_len, num_splits)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    sl = seq_lens.to(device=q.device, dtype=torch.int32).contiguous()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().qattn_decode_fp16(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, D, cap, _ptr(sl), max_seq_len,
                                            float(softmax_scale), num_splits, _ptr(workspace), ws_bytes, _ptr(out),
                                            _ptr(lse), _stream(q.device)), "qattn_decode_fp16")
    return (out, lse) if return_lse else out


def prefill_fp16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, nk: int, softmax_scale: float,
                 causal: bool = True, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 return_lse: bool = False):
    """q [B, Hq, Nq, D] fp16 against the first nk keys of k, v [B, Hkv, capacity, D] fp16."""
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    B, Hq, Nq, D = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    _check(load_library().qattn_prefill_fp16(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, D, cap, Nq, nk,
                                             float(softmax_scale), int(bool(causal)), _ptr(out), _ptr(lse),
                                             _stream(q.device)), "qattn_prefill_fp16")
    return (out, lse) if return_lse else out


# ------------------------------------------------------- progressive storage

@dataclass
class PqCache:
    """Progressive INT8 -> INT4 cache in 64-token blocks (see qattn_pq_cache):
    codes [B, Hkv, capacity, D/2] uint8, params [B, Hkv, capacity/64, 2D+16] uint8."""
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_params: torch.Tensor
    v_params: torch.Tensor
    head_dim: int
    num_kv_heads: int
    capacity: int

    @staticmethod
    def contiguous(batch, num_kv_heads, capacity, head_dim, device="cuda"):
        cap = -(-capacity // PAGE_SIZE) * PAGE_SIZE
        codes = lambda: torch.zeros(batch, num_kv_heads, cap, head_dim // 2, dtype=torch.uint8, device=device)
        params = lambda: torch.zeros(batch, num_kv_heads, cap // PAGE_SIZE, 2 * head_dim + 16, dtype=torch.uint8,
                                     device=device)
        return PqCache(codes(), codes(), params(), params(), head_dim, num_kv_heads, cap)

    def struct(self) -> PqCacheStruct:
        return PqCacheStruct(self.k_codes.data_ptr(), self.v_codes.data_ptr(), self.k_params.data_ptr(),
                             self.v_params.data_ptr(), self.head_dim, self.num_kv_heads, self.capacity)


def pq_quantize(k: torch.Tensor, v: torch.Tensor, cache: PqCache, start_block: Optional[torch.Tensor] = None) -> None:
    """k, v [B, Hkv, n, D] (fp32 or fp16, n a multiple of 64) -> n/64 blocks at start_block[b] + i."""
    if k.dtype not in (torch.float32, torch.float16) or v.dtype != k.dtype:
        raise TypeError("k and v must both be float32 or float16")
    k, v = k.contiguous(), v.contiguous()
    B, _, n, _ = k.shape
    sb = None if start_block is None else start_block.to(device=k.device, dtype=torch.int32).contiguous()
    st = cache.struct()
    dt = QATTN_F16 if k.dtype == torch.float16 else QATTN_F32
    _check(load_library().qattn_pq_quantize(_ptr(k), _ptr(v), dt, B, n, _ptr(sb), ctypes.byref(st),
                                            _stream(k.device)), "qattn_pq_quantize")


def flashq_flush_pq(buf, cache: PqCache, cache_lens: torch.Tensor) -> None:
    """Full decode buffers -> one progressive block each at cache_lens[b] (a multiple of 64)."""
    st = cache.struct()
    bs = buf.struct()
    cl = cache_lens.to(device=cache.k_codes.device, dtype=torch.int32).contiguous()
    _check(load_library().qattn_flashq_flush_pq(ctypes.byref(bs), ctypes.byref(st), _ptr(cl), cl.numel(),
                                                _stream(cache.k_codes.device)), "qattn_flashq_flush_pq")


def decode_pq_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_splits=0) -> int:
    return int(load_library().qattn_decode_pq_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                             max_seq_len, num_splits))


def decode_pq(q: torch.Tensor, cache: PqCache, seq_lens: torch.Tensor, max_seq_len: int, softmax_scale: float,
              num_splits: int = 0, workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
              lse: Optional[torch.Tensor] = None, return_lse: bool = False):
    """q [B, Hq, D] fp16 against a progressive cache -> out [B, Hq, D] fp16 (and lse)."""
    q = q.contiguous()
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if workspace is None:
        need = decode_pq_workspace_size(B, Hq, cache.num_kv_heads, D, max_seq_len, num_splits)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    sl = seq_lens.to(device=q.device, dtype=torch.int32).contiguous()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = cache.struct()
    _check(load_library().qattn_decode_pq(_ptr(q), ctypes.byref(st), _ptr(sl), B, Hq, max_seq_len,
                                          float(softmax_scale), num_splits, _ptr(workspace), ws_bytes, _ptr(out),
                                          _ptr(lse), _stream(q.device)), "qattn_decode_pq")
    return (out, lse) if return_lse else out


def combine(partial_o: torch.Tensor, partial_lse: torch.Tensor, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, return_lse: bool = False):
    """partial_o [S, R, D] fp32, partial_lse [S, R] fp32 -> out [R, D] fp16 (and lse [R])."""
    partial_o, partial_lse = partial_o.contiguous(), partial_lse.contiguous()
    S, R, D = partial_o.shape
    if out is None:
        out = torch.empty(R, D, dtype=torch.float16, device=partial_o.device)
    if lse is None and return_lse:
        lse = torch.empty(R, dtype=torch.float32, device=partial_o.device)
    _check(load_library().qattn_combine(_ptr(partial_o), _ptr(partial_lse), S, R, D, _ptr(out), _ptr(lse),
                                        _stream(partial_o.device)), "qattn_combine")
    return (out, lse) if return_lse else out


def check_wait_timeout(limit_cycles: int = 2_000_000, device="cuda") -> int:
    """Run the library's bounded-wait check on `device`; returns the QATTN_FLAG_*
    bits the check raised (FLAG_WAIT_TIMEOUT when the wait gave up as it must)."""
    flags = torch.full((1,), -1, dtype=torch.int32, device=device)
    _check(load_library().qattn_check_wait_timeout(_ptr(flags), int(limit_cycles), _stream(flags.device)),
           "qattn_check_wait_timeout")
    return int(flags.cpu().item()) & 0xFFFFFFFF


def read_device_flags(clear: bool = True) -> int:
    """Synchronise the device and return the QATTN_FLAG_* bits raised by the kernels."""
    f = ctypes.c_uint32(0)
    _check(load_library().qattn_read_device_flags(ctypes.byref(f), int(clear)), "qattn_read_device_flags")
    return int(f.value)


def headwise_plan(k: torch.Tensor, v: torch.Tensor, num_low: int, lens: Optional[torch.Tensor] = None):
    """Headwise mixed precision (qattn_headwise_plan): priorities of the kv-heads of a
    prompt's k, v [B, Hkv, n, D] (fp32 or fp16) and bits [Hkv] int32, 2 for the num_low
    lowest-priority heads and 4 for the others.  Returns (bits, priority float64)."""
    if k.dtype not in (torch.float32, torch.float16) or v.dtype != k.dtype:
        raise TypeError("k and v must both be float32 or float16")
    k, v = k.contiguous(), v.contiguous()
    B, H, n, D = k.shape
    bits = torch.empty(H, dtype=torch.int32, device=k.device)
    prio = torch.empty(H, dtype=torch.float64, device=k.device)
    ln = None if lens is None else lens.to(device=k.device, dtype=torch.int32).contiguous()
    dt = QATTN_F16 if k.dtype == torch.float16 else QATTN_F32
    _check(load_library().qattn_headwise_plan(_ptr(k), _ptr(v), dt, B, H, n, D, _ptr(ln), num_low, _ptr(bits),
                                              _ptr(prio), _stream(k.device)), "qattn_headwise_plan")
    return bits, prio


def mixed_caches(bits, batch: int, capacity: int, head_dim: int, device="cuda"):
    """The two caches of a headwise plan: (4-bit heads, 2-bit heads), each listing its
    heads' model indices in kv_head_index (None when a width has no head)."""
    b = [int(x) for x in (bits.tolist() if torch.is_tensor(bits) else bits)]
    caches = []
    for width in (4, 2):
        idx = [h for h, x in enumerate(b) if x == width]
        if not idx:
            caches.append(None)
            continue
        c = KvCache.contiguous(batch, len(idx), capacity, head_dim, device, code_bits=width)
        c.kv_head_index = torch.tensor(idx, dtype=torch.int32, device=device)
        c.model_kv_heads = len(b)
        caches.append(c)
    return tuple(caches)


def decode_mixed(q: torch.Tensor, caches, seq_lens: torch.Tensor, max_seq_len: int, softmax_scale: float,
                 num_splits: int = 0, return_lse: bool = False):
    """Decode over the caches of a headwise plan: each writes the rows of its own heads."""
    q = q.contiguous()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device) if return_lse else None
    for c in caches:
        if c is not None:
            decode(q, c, seq_lens, max_seq_len, softmax_scale, num_splits, out=out, lse=lse)
    return (out, lse) if return_lse else out
