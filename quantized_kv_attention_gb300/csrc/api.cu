// api.cu -- the C ABI declared in include/qattn.h: argument validation,
// TMA descriptor encoding, split-KV sizing and kernel dispatch.  Host code
// only; no call allocates memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/qattn.h"
#include "internal.h"

namespace qattn {

// The device status word (QATTN_FLAG_* bits), one per device that loads the
// library; kernels receive its device address.
__device__ uint32_t g_status_word;

namespace {

thread_local char t_last_error[512] = "";

qattn_status fail(qattn_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return st;
}

qattn_status cuda_fail(cudaError_t e, const char *what) {
  return fail(QATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  uint32_t *status = nullptr;
  int sms = 0;
  cudaError_t err = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

// Per-device set-up: the status word's device address and the SM count.
qattn_status device_state(DeviceState **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(QATTN_ERR_UNSUPPORTED, "device %d", dev);
  DeviceState &s = g_dev[dev];
  std::call_once(s.once, [&s, dev]() {
    s.err = cudaGetSymbolAddress(reinterpret_cast<void **>(&s.status), g_status_word);
    if (s.err == cudaSuccess) s.err = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev);
  });
  if (s.err != cudaSuccess) return cuda_fail(s.err, "device set-up");
  *out = &s;
  return QATTN_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static std::once_flag once;
  static EncodeFn fn = nullptr;
  std::call_once(once, []() {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// Prefill maps over q and out [batch*Hq, nq, D] fp16 (128B swizzle, 64
// columns per box): Q boxes of 128 rows (loads), O boxes of 32 rows (one
// warp's stores).  Rows past nq read as zero and are never written.
qattn_status prefill_maps(CUtensorMap *qmap, CUtensorMap *omap, const void *q, const void *out, int batch, int hq,
                          int nq, int head_dim) {
  EncodeFn enc = encode_fn();
  if (!enc) return fail(QATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const uint64_t heads = static_cast<uint64_t>(batch) * hq;
  if (heads > 0x7fffffffull) return fail(QATTN_ERR_UNSUPPORTED, "batch * Hq too large");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(nq), heads};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2, static_cast<cuuint64_t>(nq) * head_dim * 2};
  cuuint32_t es[3] = {1, 1, 1};
  const void *bases[2] = {q, out};
  CUtensorMap *maps[2] = {qmap, omap};
  const cuuint32_t rows[2] = {128, 32};
  for (int i = 0; i < 2; ++i) {
    cuuint32_t box[3] = {64, rows[i], 1};
    CUresult r = enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(bases[i]), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for prefill map %d", (int)r, i);
  }
  return QATTN_OK;
}

// Decode maps: codes as 3-D [heads][rows_per_head][128 B] (128B swizzle),
// scales as 2-D [heads][tokens_per_head] fp16; boxes from decode_geometry().
qattn_status decode_maps(DecodeMaps *m, const KvView &v, int batch, int warps) {
  EncodeFn enc = encode_fn();
  if (!enc) return fail(QATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const bool paged = v.page_table != nullptr;
  const DecodeGeometry geo = decode_geometry(v.head_dim, v.hkv, paged, warps);
  const uint64_t heads = paged ? static_cast<uint64_t>(v.num_pages) * v.hkv : static_cast<uint64_t>(batch) * v.hkv;
  const uint64_t tokens = paged ? kPage : static_cast<uint64_t>(v.capacity);
  // code bytes per token: D/2 (INT4) or 52 (INT3, D = 128); INT3 stages are
  // read with plain word loads, so their boxes are not swizzled
  const uint64_t tok_bytes = v.bits == 3 ? 52 : static_cast<uint64_t>(v.head_dim * v.bits / 8);
  const uint64_t rows = tokens * tok_bytes / 128;
  const cuuint32_t box_rows = v.bits != 4 ? static_cast<cuuint32_t>(geo.tokens_per_stage * tok_bytes / 128)
                                          : static_cast<cuuint32_t>(geo.box_rows);
  if (heads > 0x7fffffffull || rows > 0x7fffffffull) return fail(QATTN_ERR_UNSUPPORTED, "cache too large");
  const void *bases[4] = {v.k_codes, v.v_codes, v.k_scales, v.v_scales};
  CUtensorMap *outs[4] = {&m->k, &m->v, &m->ks, &m->vs};
  for (int i = 0; i < 4; ++i) {
    CUresult r;
    if (i < 2) {
      cuuint64_t dims[3] = {128, rows, heads};
      cuuint64_t strides[2] = {128, rows * 128};
      cuuint32_t box[3] = {128, box_rows, static_cast<cuuint32_t>(geo.box_heads)};
      cuuint32_t es[3] = {1, 1, 1};
      r = enc(outs[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(bases[i]), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, v.bits == 3 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      cuuint64_t dims[2] = {tokens, heads};
      cuuint64_t strides[1] = {tokens * 2};
      cuuint32_t box[2] = {static_cast<cuuint32_t>(geo.box_tokens), static_cast<cuuint32_t>(geo.box_heads)};
      cuuint32_t es[2] = {1, 1};
      r = enc(outs[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(bases[i]), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return fail(QATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for decode map %d", (int)r, i);
  }
  return QATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by every call that reads or writes the cache.
qattn_status check_cache(const qattn_kv_cache *c, int batch, KvView *v, uint64_t *code_bytes) {
  if (!c) return fail(QATTN_ERR_INVALID_ARG, "cache is NULL");
  if (!c->k_codes || !c->k_scales || !c->v_codes || !c->v_scales)
    return fail(QATTN_ERR_INVALID_ARG, "cache has a NULL code or scale pointer");
  if (!aligned16(c->k_codes) || !aligned16(c->v_codes) || !aligned16(c->k_scales) || !aligned16(c->v_scales))
    return fail(QATTN_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(QATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", c->head_dim);
  if (c->num_kv_heads <= 0) return fail(QATTN_ERR_INVALID_ARG, "num_kv_heads %d", c->num_kv_heads);
  v->k_codes = c->k_codes, v->k_scales = c->k_scales, v->v_codes = c->v_codes, v->v_scales = c->v_scales;
  v->page_table = c->page_table;
  v->hkv = c->num_kv_heads;
  v->head_dim = c->head_dim;
  if (c->code_bits != 0 && c->code_bits != 4 && c->code_bits != 3 && c->code_bits != 2)
    return fail(QATTN_ERR_INVALID_ARG, "code_bits %d (0 or 4: INT4, 3: INT3, 2: INT2)", c->code_bits);
  v->bits = c->code_bits == 0 ? 4 : c->code_bits;
  if (v->bits != 4 && (c->page_table || c->head_dim != 128))
    return fail(QATTN_ERR_UNSUPPORTED, "INT%d needs a contiguous cache with head_dim 128", v->bits);
  v->head_map = c->kv_head_index;
  v->model_hkv = c->num_kv_heads;
  if (c->kv_head_index) {
    if (c->page_table) return fail(QATTN_ERR_UNSUPPORTED, "kv_head_index with a paged cache");
    if (c->model_kv_heads < c->num_kv_heads)
      return fail(QATTN_ERR_INVALID_ARG, "model_kv_heads %d < num_kv_heads %d", c->model_kv_heads, c->num_kv_heads);
    v->model_hkv = c->model_kv_heads;
  }
  const uint64_t row_bytes = v->bits == 3 ? 52 : static_cast<uint64_t>(c->head_dim * v->bits / 8);
  v->capacity = 0, v->num_pages = 0, v->max_pages = 0;
  if (c->page_table) {
    if (c->page_size != QATTN_PAGE_SIZE)
      return fail(QATTN_ERR_UNSUPPORTED, "page_size %d (supported: %d)", c->page_size, QATTN_PAGE_SIZE);
    if (c->num_pages <= 0 || c->max_pages_per_seq <= 0)
      return fail(QATTN_ERR_INVALID_ARG, "paged cache needs num_pages > 0 and max_pages_per_seq > 0");
    v->num_pages = c->num_pages;
    v->max_pages = c->max_pages_per_seq;
    *code_bytes = static_cast<uint64_t>(c->num_pages) * c->num_kv_heads * kPage * row_bytes;
  } else {
    if (c->capacity <= 0 || c->capacity % kPage)
      return fail(QATTN_ERR_UNSUPPORTED, "capacity %lld must be a positive multiple of %d",
                  (long long)c->capacity, kPage);
    v->capacity = c->capacity;
    *code_bytes = static_cast<uint64_t>(batch) * c->num_kv_heads * c->capacity * row_bytes;
  }
  return QATTN_OK;
}

// Number of balanced key ranges (one persistent CTA each) for a decode call:
// one per SM by default, never more than there can be stages.
int plan_ctas(int batch, int hkv, int head_dim, int max_len, int requested, int sms, bool paged, int warps) {
  const DecodeGeometry geo = decode_geometry(head_dim, hkv, paged, warps);
  const int64_t stages = static_cast<int64_t>(batch) * geo.groups *
                         ((static_cast<int64_t>(max_len) + geo.tokens_per_stage - 1) / geo.tokens_per_stage);
  int64_t n = requested > 0 ? requested : sms;
  if (n > stages) n = stages;
  if (n > QATTN_MAX_SPLITS) n = QATTN_MAX_SPLITS;
  if (n < 1) n = 1;
  return static_cast<int>(n);
}

// partial_o [2*ctas, rows, D] fp32, padded to 256 bytes, then partial_lse
// [2*ctas, rows]; rows = kv-heads per stage * G.
size_t workspace_bytes(int ctas, int rows, int head_dim) {
  const size_t o = static_cast<size_t>(2) * ctas * rows * head_dim * sizeof(float);
  return (o + 255) / 256 * 256 + static_cast<size_t>(2) * ctas * rows * sizeof(float);
}

// Paged pools stream up to 4 adjacent kv-heads per stage, so Hkv must split evenly.
bool hkv_supported(int hkv, bool paged) {
  return hkv > 0 && (!paged || hkv == 1 || hkv == 2 || hkv % 4 == 0);
}

}  // namespace

// Lets other translation units of the library report a failure through
// qattn_last_error().
void record_error(const char *msg) { snprintf(t_last_error, sizeof(t_last_error), "%s", msg); }

}  // namespace qattn

using namespace qattn;

extern "C" {

qattn_status qattn_quantize_kv(const void *k, const void *v, qattn_dtype x_dtype, int32_t batch,
                               int32_t n, const int32_t *start_pos, const qattn_kv_cache *cache,
                               qattn_stream_t stream) {
  if (batch < 0 || n < 0) return fail(QATTN_ERR_INVALID_ARG, "batch %d, n %d", batch, n);
  if (x_dtype != QATTN_F32 && x_dtype != QATTN_F16) return fail(QATTN_ERR_INVALID_ARG, "x_dtype %d", (int)x_dtype);
  KvView view;
  uint64_t code_bytes = 0;
  qattn_status st = check_cache(cache, batch, &view, &code_bytes);
  if (st != QATTN_OK) return st;
  if (batch == 0 || n == 0) return QATTN_OK;
  if (!k || !v) return fail(QATTN_ERR_INVALID_ARG, "k or v is NULL");
  if (!aligned16(k) || !aligned16(v)) return fail(QATTN_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_quantize(k, v, x_dtype == QATTN_F16, batch, n, start_pos, view, ds->status, ds->sms,
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "quantize launch");
}

qattn_status qattn_headwise_plan(const void *k, const void *v, qattn_dtype x_dtype, int32_t batch,
                                 int32_t num_kv_heads, int32_t n, int32_t head_dim, const int32_t *lens,
                                 int32_t num_low, int32_t *bits, double *priority, qattn_stream_t stream) {
  if (batch < 0 || batch > QATTN_MAX_BATCH || n < 0)
    return fail(QATTN_ERR_INVALID_ARG, "batch %d, n %d", batch, n);
  if (x_dtype != QATTN_F32 && x_dtype != QATTN_F16) return fail(QATTN_ERR_INVALID_ARG, "x_dtype %d", (int)x_dtype);
  if (head_dim != 64 && head_dim != 128) return fail(QATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (num_kv_heads <= 0 || num_kv_heads > headwise_max_heads())
    return fail(QATTN_ERR_UNSUPPORTED, "num_kv_heads %d (1..%d)", num_kv_heads, headwise_max_heads());
  if (num_low < 0 || num_low > num_kv_heads)
    return fail(QATTN_ERR_INVALID_ARG, "num_low %d (0..%d)", num_low, num_kv_heads);
  if (!bits) return fail(QATTN_ERR_INVALID_ARG, "bits is NULL");
  if (batch > 0 && n > 0) {
    if (!k || !v) return fail(QATTN_ERR_INVALID_ARG, "k or v is NULL");
    if (static_cast<int64_t>((n + 255) / 256) * batch * num_kv_heads > 0x7fffffffLL)
      return fail(QATTN_ERR_UNSUPPORTED, "batch * Hkv * n too large");
  }
  DeviceState *ds;
  qattn_status st = device_state(&ds);
  if (st != QATTN_OK) return st;
  cudaError_t e = launch_headwise_plan(k, v, x_dtype == QATTN_F16, batch, num_kv_heads, batch > 0 ? n : 0,
                                       head_dim, lens, num_low, bits, priority,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "headwise plan launch");
}

qattn_status qattn_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t max_seq_len, int32_t num_splits, int32_t paged, int32_t code_bits,
                               int32_t has_kv_head_index, int32_t *warps, int32_t *ctas, int32_t *cluster) {
  if (batch <= 0 || batch > QATTN_MAX_BATCH || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > QATTN_MAX_GROUP || max_seq_len < 0 ||
      num_splits < 0 || num_splits > QATTN_MAX_SPLITS || (head_dim != 64 && head_dim != 128) ||
      (code_bits != 4 && code_bits != 3 && code_bits != 2) || !hkv_supported(num_kv_heads, paged != 0))
    return fail(QATTN_ERR_INVALID_ARG, "decode plan: invalid sizes");
  DeviceState *ds;
  qattn_status st = device_state(&ds);
  if (st != QATTN_OK) return st;
  const int w = decode_layout(batch, num_kv_heads, max_seq_len, paged != 0, num_splits > 0 ? num_splits : ds->sms);
  int n = plan_ctas(batch, num_kv_heads, head_dim, max_seq_len, num_splits, ds->sms, paged != 0, w);
  const int S = decode_cluster(head_dim, w, code_bits, num_splits == 0, paged != 0, has_kv_head_index != 0, batch,
                               num_kv_heads, max_seq_len, ds->sms);
  if (S > 0) n = batch * decode_geometry(head_dim, num_kv_heads, false, w).groups * S;
  if (warps) *warps = w;
  if (ctas) *ctas = n;
  if (cluster) *cluster = S;
  return QATTN_OK;
}

size_t qattn_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_seq_len, int32_t num_splits) {
  if (batch <= 0 || batch > QATTN_MAX_BATCH || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > QATTN_MAX_GROUP || max_seq_len < 0 ||
      num_kv_heads <= 0 ||
      num_splits < 0 || num_splits > QATTN_MAX_SPLITS || (head_dim != 64 && head_dim != 128))
    return 0;
  // The automatic split count follows the current device's SM count, cached
  // by the per-device set-up; without a usable device the answer assumes
  // 152 SMs.  Only an error raised by this query is cleared from the
  // runtime, never one pending from the caller's own work.
  int sms = 152;
  if (num_splits == 0) {
    DeviceState *ds = nullptr;
    if (device_state(&ds) == QATTN_OK && ds->sms > 0)
      sms = ds->sms;
    else
      cudaGetLastError();
  }
  // the larger of the two cache layouts' needs (the call does not say which one)
  size_t need = 0;
  // (and of both CTA layouts, so that the answer never depends on the choice)
  for (int paged = 0; paged < 2; ++paged) {
    if (paged && !hkv_supported(num_kv_heads, true)) continue;
    for (int warps = 8; warps <= 12; warps += 4) {
      if (paged && warps != 8) continue;
      const int ctas = plan_ctas(batch, num_kv_heads, head_dim, max_seq_len, num_splits, sms, paged != 0, warps);
      const DecodeGeometry geo = decode_geometry(head_dim, num_kv_heads, paged != 0, warps);
      const size_t n = workspace_bytes(ctas, geo.heads_per_stage * (num_q_heads / num_kv_heads), head_dim);
      if (n > need) need = n;
    }
  }
  return need;
}

}  // extern "C"

namespace qattn {
namespace {

// qattn_decode and qattn_decode_append: the latter passes the new rows.
qattn_status decode_impl(const uint16_t *q, const void *k_new, const void *v_new, bool new_fp16,
                         const qattn_kv_cache *cache, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                         int32_t max_seq_len, float softmax_scale, int32_t num_splits, void *workspace,
                         size_t workspace_size, uint16_t *out, float *lse, qattn_stream_t stream) {
  if (batch < 0 || num_q_heads <= 0 || max_seq_len < 0)
    return fail(QATTN_ERR_INVALID_ARG, "batch %d, num_q_heads %d, max_seq_len %d", batch, num_q_heads, max_seq_len);
  if (batch > QATTN_MAX_BATCH) return fail(QATTN_ERR_UNSUPPORTED, "batch %d > %d", batch, QATTN_MAX_BATCH);
  if (num_splits < 0 || num_splits > QATTN_MAX_SPLITS)
    return fail(QATTN_ERR_INVALID_ARG, "num_splits %d (0..%d)", num_splits, QATTN_MAX_SPLITS);
  KvView view;
  uint64_t code_bytes = 0;
  qattn_status st = check_cache(cache, batch, &view, &code_bytes);
  if (st != QATTN_OK) return st;
  if (num_q_heads % view.model_hkv)
    return fail(QATTN_ERR_INVALID_ARG, "Hq %d is not a multiple of the model's Hkv %d", num_q_heads, view.model_hkv);
  if (num_q_heads / view.model_hkv > QATTN_MAX_GROUP)
    return fail(QATTN_ERR_UNSUPPORTED, "group size %d > %d", num_q_heads / view.model_hkv, QATTN_MAX_GROUP);
  if (!hkv_supported(view.hkv, view.page_table != nullptr))
    return fail(QATTN_ERR_UNSUPPORTED, "paged num_kv_heads %d (supported: 1, 2 or a multiple of 4)", view.hkv);
  if (batch == 0) return QATTN_OK;
  if (!q || !seq_lens || !out) return fail(QATTN_ERR_INVALID_ARG, "q, seq_lens or out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(QATTN_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(QATTN_ERR_INVALID_ARG, "k_new and v_new: both or neither");
  if (view.bits != 4 && k_new) return fail(QATTN_ERR_UNSUPPORTED, "qattn_decode_append on an INT%d cache", view.bits);
  if (view.head_map && k_new) return fail(QATTN_ERR_UNSUPPORTED, "qattn_decode_append with kv_head_index");
  if (k_new && (!aligned16(k_new) || !aligned16(v_new)))
    return fail(QATTN_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  const int G = num_q_heads / view.model_hkv;
  const int64_t stage_limit = view.page_table ? view.max_pages : view.capacity / kPage;
  if (static_cast<int64_t>(batch) * view.hkv * stage_limit >= (int64_t(1) << 31))
    return fail(QATTN_ERR_UNSUPPORTED, "batch * Hkv * cached stages exceeds 2^31");
  const bool paged = view.page_table != nullptr;
  const int warps = decode_layout(batch, view.hkv, max_seq_len, paged,
                                                        num_splits > 0 ? num_splits : ds->sms);
  const int ctas = plan_ctas(batch, view.hkv, view.head_dim, max_seq_len, num_splits, ds->sms, paged, warps);
  const DecodeGeometry geo = decode_geometry(view.head_dim, view.hkv, paged, warps);
  const int slot_rows = geo.heads_per_stage * G;
  const size_t need = workspace_bytes(ctas, slot_rows, view.head_dim);
  if (!workspace || workspace_size < need || !aligned16(workspace))
    return fail(QATTN_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, %zu given", need,
                workspace ? workspace_size : (size_t)0);
  DecodeMaps maps;
  if ((st = decode_maps(&maps, view, batch, warps)) != QATTN_OK) return st;

  DecodeArgs a;
  a.q = q, a.seq_lens = seq_lens, a.out = out, a.lse = lse;
  a.partial_o = static_cast<float *>(workspace);
  const size_t o_bytes = static_cast<size_t>(2) * ctas * slot_rows * view.head_dim * sizeof(float);
  a.partial_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + (o_bytes + 255) / 256 * 256);
  a.k_new = k_new, a.v_new = v_new, a.new_fp16 = new_fp16 ? 1 : 0;
  a.max_len = max_seq_len;
  a.batch = batch, a.hq = num_q_heads, a.ctas = ctas, a.warps = warps;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.auto_splits = num_splits == 0, a.sms = ds->sms, a.cluster = 0;
  cudaError_t e = launch_decode(a, view, maps, ds->status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "decode launch");
}

}  // namespace
}  // namespace qattn

extern "C" {

qattn_status qattn_decode(const uint16_t *q, const qattn_kv_cache *cache, const int32_t *seq_lens,
                          int32_t batch, int32_t num_q_heads, int32_t max_seq_len,
                          float softmax_scale, int32_t num_splits, void *workspace,
                          size_t workspace_size, uint16_t *out, float *lse, qattn_stream_t stream) {
  return decode_impl(q, nullptr, nullptr, false, cache, seq_lens, batch, num_q_heads, max_seq_len, softmax_scale,
                     num_splits, workspace, workspace_size, out, lse, stream);
}

qattn_status qattn_decode_append(const uint16_t *q, const void *k_new, const void *v_new, qattn_dtype x_dtype,
                                 const qattn_kv_cache *cache, const int32_t *seq_lens, int32_t batch,
                                 int32_t num_q_heads, int32_t max_seq_len, float softmax_scale,
                                 int32_t num_splits, void *workspace, size_t workspace_size, uint16_t *out,
                                 float *lse, qattn_stream_t stream) {
  if (x_dtype != QATTN_F32 && x_dtype != QATTN_F16) return fail(QATTN_ERR_INVALID_ARG, "x_dtype %d", (int)x_dtype);
  if (batch > 0 && (!k_new || !v_new)) return fail(QATTN_ERR_INVALID_ARG, "k_new or v_new is NULL");
  return decode_impl(q, k_new, v_new, x_dtype == QATTN_F16, cache, seq_lens, batch, num_q_heads, max_seq_len,
                     softmax_scale, num_splits, workspace, workspace_size, out, lse, stream);
}

}  // extern "C"

namespace qattn {
namespace {

// Validates a decode buffer (and, when given, that it matches the cache).
qattn_status check_flashq(const qattn_flashq_buffer *b, int batch, FlashqView *v) {
  if (!b) return fail(QATTN_ERR_INVALID_ARG, "flashq buffer is NULL");
  if (batch < 0 || batch > QATTN_MAX_BATCH) return fail(QATTN_ERR_INVALID_ARG, "batch %d", batch);
  if (b->head_dim != 64 && b->head_dim != 128) return fail(QATTN_ERR_UNSUPPORTED, "head_dim %d", b->head_dim);
  if (b->num_kv_heads < 1 || b->num_kv_heads > 64)
    return fail(QATTN_ERR_INVALID_ARG, "num_kv_heads %d (1..64)", b->num_kv_heads);
  if (!b->k_codes || !b->v_codes || !b->k_scale || !b->v_scale || !b->k_range || !b->v_range || !b->count)
    return fail(QATTN_ERR_INVALID_ARG, "a flashq buffer pointer is NULL");
  if (!aligned16(b->k_codes) || !aligned16(b->v_codes))
    return fail(QATTN_ERR_INVALID_ARG, "flashq codes must be 16-byte aligned");
  v->k_codes = b->k_codes, v->v_codes = b->v_codes, v->k_scale = b->k_scale, v->v_scale = b->v_scale;
  v->k_range = b->k_range, v->v_range = b->v_range, v->count = b->count;
  v->hkv = b->num_kv_heads, v->head_dim = b->head_dim;
  return QATTN_OK;
}

qattn_status check_flashq_cache(const qattn_flashq_buffer *b, const qattn_kv_cache *cache,
                                const int32_t *cache_lens, int batch, FlashqView *fv, KvView *kv) {
  qattn_status st = check_flashq(b, batch, fv);
  if (st != QATTN_OK) return st;
  uint64_t code_bytes = 0;
  if ((st = check_cache(cache, batch, kv, &code_bytes)) != QATTN_OK) return st;
  if (kv->bits != 4) return fail(QATTN_ERR_UNSUPPORTED, "the decode buffer on an INT%d cache", kv->bits);
  if (kv->head_map) return fail(QATTN_ERR_UNSUPPORTED, "the decode buffer with kv_head_index");
  if (kv->head_dim != fv->head_dim || kv->hkv != fv->hkv)
    return fail(QATTN_ERR_INVALID_ARG, "buffer (D %d, Hkv %d) and cache (D %d, Hkv %d) differ", fv->head_dim,
                fv->hkv, kv->head_dim, kv->hkv);
  if (batch > 0 && !cache_lens) return fail(QATTN_ERR_INVALID_ARG, "cache_lens is NULL");
  return QATTN_OK;
}

}  // namespace
}  // namespace qattn

extern "C" {

qattn_status qattn_flashq_init(const qattn_flashq_buffer *buf, const qattn_kv_cache *cache,
                               const int32_t *cache_lens, int32_t batch, qattn_stream_t stream) {
  FlashqView fv;
  KvView kv;
  qattn_status st = check_flashq_cache(buf, cache, cache_lens, batch, &fv, &kv);
  if (st != QATTN_OK || batch == 0) return st;
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_flashq_init(fv, kv, cache_lens, batch, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "flashq init launch");
}

qattn_status qattn_flashq_append(const void *k_new, const void *v_new, qattn_dtype x_dtype,
                                 const qattn_flashq_buffer *buf, int32_t batch, qattn_stream_t stream) {
  if (x_dtype != QATTN_F32 && x_dtype != QATTN_F16) return fail(QATTN_ERR_INVALID_ARG, "x_dtype %d", (int)x_dtype);
  FlashqView fv;
  qattn_status st = check_flashq(buf, batch, &fv);
  if (st != QATTN_OK || batch == 0) return st;
  if (!k_new || !v_new) return fail(QATTN_ERR_INVALID_ARG, "k_new or v_new is NULL");
  if (!aligned16(k_new) || !aligned16(v_new)) return fail(QATTN_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_flashq_append(k_new, v_new, x_dtype == QATTN_F16, fv, batch, ds->status,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "flashq append launch");
}

qattn_status qattn_flashq_attend(const uint16_t *q, const qattn_flashq_buffer *buf, int32_t batch,
                                 int32_t num_q_heads, float softmax_scale, uint16_t *out, float *lse,
                                 qattn_stream_t stream) {
  FlashqView fv;
  qattn_status st = check_flashq(buf, batch, &fv);
  if (st != QATTN_OK) return st;
  if (num_q_heads <= 0 || num_q_heads % fv.hkv)
    return fail(QATTN_ERR_INVALID_ARG, "Hq %d is not a positive multiple of Hkv %d", num_q_heads, fv.hkv);
  if (num_q_heads / fv.hkv > QATTN_MAX_GROUP)
    return fail(QATTN_ERR_UNSUPPORTED, "group size %d > %d", num_q_heads / fv.hkv, QATTN_MAX_GROUP);
  if (batch == 0) return QATTN_OK;
  if (!q || !out || !lse) return fail(QATTN_ERR_INVALID_ARG, "q, out or lse is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(QATTN_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_flashq_attend(q, fv, batch, num_q_heads, softmax_scale * 1.4426950408889634f, out, lse,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "flashq attend launch");
}

qattn_status qattn_flashq_flush(const qattn_flashq_buffer *buf, const qattn_kv_cache *cache,
                                const int32_t *cache_lens, int32_t batch, qattn_stream_t stream) {
  FlashqView fv;
  KvView kv;
  qattn_status st = check_flashq_cache(buf, cache, cache_lens, batch, &fv, &kv);
  if (st != QATTN_OK || batch == 0) return st;
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_flashq_flush(fv, kv, cache_lens, batch, ds->status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "flashq flush launch");
}

qattn_status qattn_prefill(const uint16_t *q, const qattn_kv_cache *cache, int32_t batch,
                           int32_t num_q_heads, int32_t nq, int32_t nk, float softmax_scale,
                           int32_t causal, uint16_t *out, float *lse, qattn_stream_t stream) {
  if (batch < 0 || num_q_heads <= 0 || nq < 0 || nk < 0 || (causal != 0 && causal != 1))
    return fail(QATTN_ERR_INVALID_ARG, "batch %d, Hq %d, nq %d, nk %d, causal %d", batch, num_q_heads, nq, nk, causal);
  KvView view;
  uint64_t code_bytes = 0;
  qattn_status st = check_cache(cache, batch, &view, &code_bytes);
  if (st != QATTN_OK) return st;
  if (view.bits != 4) return fail(QATTN_ERR_UNSUPPORTED, "qattn_prefill on an INT%d cache", view.bits);
  if (view.head_map) return fail(QATTN_ERR_UNSUPPORTED, "qattn_prefill with kv_head_index");

  if (num_q_heads % view.hkv) return fail(QATTN_ERR_INVALID_ARG, "Hq %d is not a multiple of Hkv %d", num_q_heads, view.hkv);
  if (nq > nk) return fail(QATTN_ERR_INVALID_ARG, "nq %d > nk %d", nq, nk);
  const int64_t limit = view.page_table ? static_cast<int64_t>(view.max_pages) * kPage : view.capacity;
  if (nk > limit)
    return fail(QATTN_ERR_INVALID_ARG, "nk %d > the cache's %lld tokens per sequence", nk, (long long)limit);
  if (batch == 0 || nq == 0) return QATTN_OK;
  if (!q || !out) return fail(QATTN_ERR_INVALID_ARG, "q or out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(QATTN_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  CUtensorMap qmap, omap;
  if ((st = prefill_maps(&qmap, &omap, q, out, batch, num_q_heads, nq, view.head_dim)) != QATTN_OK) return st;
  PrefillArgs a;
  a.q = q, a.out = out, a.lse = lse;
  a.batch = batch, a.hq = num_q_heads, a.nq = nq, a.nk = nk, a.causal = causal;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  cudaError_t e = launch_prefill(a, view, qmap, omap, ds->status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "prefill launch");
}

qattn_status qattn_combine(const float *partial_o, const float *partial_lse, int32_t num_splits,
                           int64_t rows, int32_t head_dim, uint16_t *out, float *lse,
                           qattn_stream_t stream) {
  if (num_splits < 1 || num_splits > QATTN_MAX_SPLITS)
    return fail(QATTN_ERR_INVALID_ARG, "num_splits %d (1..%d)", num_splits, QATTN_MAX_SPLITS);
  if (rows < 0 || rows > 0x7fffffffLL) return fail(QATTN_ERR_INVALID_ARG, "rows %lld", (long long)rows);
  if (head_dim != 64 && head_dim != 128) return fail(QATTN_ERR_UNSUPPORTED, "head_dim %d", head_dim);
  if (rows == 0) return QATTN_OK;
  if (!partial_o || !partial_lse || !out) return fail(QATTN_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(partial_o) || !aligned16(out)) return fail(QATTN_ERR_INVALID_ARG, "partial_o and out must be 16-byte aligned");
  cudaError_t e = launch_combine(partial_o, partial_lse, num_splits, rows, head_dim, out, lse, false,
                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "combine launch");
}

qattn_status qattn_read_device_flags(uint32_t *flags, int32_t clear) {
  if (!flags) return fail(QATTN_ERR_INVALID_ARG, "flags is NULL");
  DeviceState *ds;
  qattn_status st = device_state(&ds);
  if (st != QATTN_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(flags, ds->status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(ds->status, 0, sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "status word");
}

const char *qattn_status_string(qattn_status status) {
  switch (status) {
    case QATTN_OK: return "ok";
    case QATTN_ERR_INVALID_ARG: return "invalid argument";
    case QATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case QATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case QATTN_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char *qattn_last_error(void) { return t_last_error; }

// ------------------------------------------------------ comparison paths

qattn_status qattn_dequantize_kv(const qattn_kv_cache *cache, int32_t batch, int32_t n, uint16_t *k_out,
                                 uint16_t *v_out, qattn_stream_t stream) {
  if (batch < 0 || n < 0) return fail(QATTN_ERR_INVALID_ARG, "batch %d, n %d", batch, n);
  KvView view;
  uint64_t code_bytes = 0;
  qattn_status st = check_cache(cache, batch, &view, &code_bytes);
  if (st != QATTN_OK) return st;
  if (view.bits != 4) return fail(QATTN_ERR_UNSUPPORTED, "qattn_dequantize_kv on an INT%d cache", view.bits);
  if (view.head_map) return fail(QATTN_ERR_UNSUPPORTED, "qattn_dequantize_kv with kv_head_index");
  const int64_t limit = view.page_table ? static_cast<int64_t>(view.max_pages) * kPage : view.capacity;
  if (n > limit) return fail(QATTN_ERR_INVALID_ARG, "n %d exceeds the cache's %lld tokens", n, (long long)limit);
  if (batch == 0 || n == 0) return QATTN_OK;
  if (!k_out || !v_out) return fail(QATTN_ERR_INVALID_ARG, "k_out or v_out is NULL");
  if (!aligned16(k_out) || !aligned16(v_out)) return fail(QATTN_ERR_INVALID_ARG, "k_out and v_out must be 16-byte aligned");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_dequantize(view, batch, n, k_out, v_out, ds->status, ds->sms,
                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "dequantize launch");
}

}  // extern "C"

namespace qattn {
namespace {

// Key ranges of an fp16 decode: the requested count, or one CTA per SM over
// all (sequence, kv-head) pairs; ranges of a multiple of 64 tokens.
void decode16_plan(int batch, int hkv, int max_len, int requested, int sms, int *splits, int *chunk) {
  const int64_t tiles = (static_cast<int64_t>(max_len) + 63) / 64;
  int64_t n = requested > 0 ? requested : max(1, sms / max(1, batch * hkv));
  n = min(n, max(tiles, static_cast<int64_t>(1)));
  n = min(n, static_cast<int64_t>(QATTN_MAX_SPLITS));
  const int64_t per = (tiles + n - 1) / n;  // tiles per range
  *chunk = static_cast<int>(max(per, static_cast<int64_t>(1)) * 64);
  *splits = static_cast<int>(max(static_cast<int64_t>(1), (static_cast<int64_t>(max_len) + *chunk - 1) / *chunk));
}

size_t decode16_workspace(int batch, int hq, int head_dim, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(splits) * batch * hq;
  return (rows * head_dim * 4 + 255) / 256 * 256 + rows * 4;
}

// An fp16 cache [heads][capacity][D] read as 3-D [heads][extent][D] (tokens
// at or past `extent` read as zero), boxes of 64 columns x box_tokens.
qattn_status fp16_cache_map(CUtensorMap *m, const void *base, int64_t heads, int64_t capacity, int64_t extent,
                            int head_dim, int box_tokens) {
  EncodeFn enc = encode_fn();
  if (!enc) return fail(QATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(extent),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2, static_cast<cuuint64_t>(capacity) * head_dim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_tokens), 1}, es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for an fp16 cache", (int)r);
  return QATTN_OK;
}

}  // namespace
}  // namespace qattn

extern "C" {

size_t qattn_decode_fp16_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_seq_len, int32_t num_splits) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
      num_q_heads / num_kv_heads > QATTN_MAX_GROUP || max_seq_len < 0 || num_splits < 0 ||
      num_splits > QATTN_MAX_SPLITS || (head_dim != 64 && head_dim != 128))
    return 0;
  int sms = 152;
  if (num_splits == 0) {
    DeviceState *ds = nullptr;
    if (device_state(&ds) == QATTN_OK && ds->sms > 0)
      sms = ds->sms;
    else
      cudaGetLastError();
  }
  int splits = 1, chunk = 64;
  decode16_plan(batch, num_kv_heads, max_seq_len, num_splits, sms, &splits, &chunk);
  return decode16_workspace(batch, num_q_heads, head_dim, splits);
}

qattn_status qattn_decode_fp16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int32_t batch,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t capacity,
                               const int32_t *seq_lens, int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                               void *workspace, size_t workspace_bytes, uint16_t *out, float *lse,
                               qattn_stream_t stream) {
  if (batch < 0 || batch > QATTN_MAX_BATCH || num_q_heads <= 0 || num_kv_heads <= 0 || max_seq_len < 0)
    return fail(QATTN_ERR_INVALID_ARG, "batch %d, Hq %d, Hkv %d, max_seq_len %d", batch, num_q_heads, num_kv_heads,
                max_seq_len);
  if (num_q_heads % num_kv_heads) return fail(QATTN_ERR_INVALID_ARG, "Hq %d is not a multiple of Hkv %d", num_q_heads, num_kv_heads);
  if (num_q_heads / num_kv_heads > QATTN_MAX_GROUP)
    return fail(QATTN_ERR_UNSUPPORTED, "group size %d > %d", num_q_heads / num_kv_heads, QATTN_MAX_GROUP);
  if (head_dim != 64 && head_dim != 128) return fail(QATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (capacity <= 0 || capacity > 0x7fffffffLL) return fail(QATTN_ERR_INVALID_ARG, "capacity %lld", (long long)capacity);
  if (num_splits < 0 || num_splits > QATTN_MAX_SPLITS)
    return fail(QATTN_ERR_INVALID_ARG, "num_splits %d (0..%d)", num_splits, QATTN_MAX_SPLITS);
  if (batch == 0) return QATTN_OK;
  if (!q || !k || !v || !seq_lens || !out) return fail(QATTN_ERR_INVALID_ARG, "q, k, v, seq_lens or out is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(QATTN_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
  if (static_cast<int64_t>(batch) * num_kv_heads > 65535)
    return fail(QATTN_ERR_UNSUPPORTED, "batch * Hkv %d > 65535", batch * num_kv_heads);
  DeviceState *ds;
  qattn_status st = device_state(&ds);
  if (st != QATTN_OK) return st;
  Decode16Args a;
  decode16_plan(batch, num_kv_heads, max_seq_len, num_splits, ds->sms, &a.splits, &a.chunk);
  const size_t need = decode16_workspace(batch, num_q_heads, head_dim, a.splits);
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return fail(QATTN_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, %zu given", need,
                workspace ? workspace_bytes : (size_t)0);
  CUtensorMap kmap, vmap;
  const int64_t heads = static_cast<int64_t>(batch) * num_kv_heads;
  if ((st = fp16_cache_map(&kmap, k, heads, capacity, capacity, head_dim, 64)) != QATTN_OK) return st;
  if ((st = fp16_cache_map(&vmap, v, heads, capacity, capacity, head_dim, 64)) != QATTN_OK) return st;
  a.q = q, a.seq_lens = seq_lens, a.out = out, a.lse = lse;
  a.partial_o = static_cast<float *>(workspace);
  const size_t rows = static_cast<size_t>(a.splits) * batch * num_q_heads;
  a.partial_lse = need ? reinterpret_cast<float *>(static_cast<char *>(workspace) + (rows * head_dim * 4 + 255) / 256 * 256)
                       : nullptr;
  a.batch = batch, a.hq = num_q_heads, a.hkv = num_kv_heads, a.head_dim = head_dim;
  a.capacity = capacity;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  cudaError_t e = launch_decode16(a, kmap, vmap, ds->status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "fp16 decode launch");
}

}  // extern "C"

namespace qattn {
namespace {

// Validates a progressive cache (batch sequences).
qattn_status check_pq(const qattn_pq_cache *c, PqView *v) {
  if (!c) return fail(QATTN_ERR_INVALID_ARG, "progressive cache is NULL");
  if (!c->k_codes || !c->v_codes || !c->k_params || !c->v_params)
    return fail(QATTN_ERR_INVALID_ARG, "progressive cache has a NULL pointer");
  if (!aligned16(c->k_codes) || !aligned16(c->v_codes) || !aligned16(c->k_params) || !aligned16(c->v_params))
    return fail(QATTN_ERR_INVALID_ARG, "progressive cache pointers must be 16-byte aligned");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(QATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", c->head_dim);
  if (c->num_kv_heads <= 0) return fail(QATTN_ERR_INVALID_ARG, "num_kv_heads %d", c->num_kv_heads);
  if (c->capacity <= 0 || c->capacity % kPage || c->capacity > 0x7fffffffLL)
    return fail(QATTN_ERR_INVALID_ARG, "capacity %lld must be a positive multiple of 64", (long long)c->capacity);
  v->k_codes = c->k_codes, v->v_codes = c->v_codes, v->k_params = c->k_params, v->v_params = c->v_params;
  v->capacity = c->capacity, v->hkv = c->num_kv_heads, v->head_dim = c->head_dim;
  return QATTN_OK;
}

}  // namespace
}  // namespace qattn

extern "C" {

qattn_status qattn_pq_quantize(const void *k, const void *v, qattn_dtype x_dtype, int32_t batch, int32_t n,
                               const int32_t *start_block, const qattn_pq_cache *cache, qattn_stream_t stream) {
  if (batch < 0 || n < 0 || n % kPage) return fail(QATTN_ERR_INVALID_ARG, "batch %d, n %d (a multiple of 64)", batch, n);
  if (x_dtype != QATTN_F32 && x_dtype != QATTN_F16) return fail(QATTN_ERR_INVALID_ARG, "x_dtype %d", (int)x_dtype);
  PqView view;
  qattn_status st = check_pq(cache, &view);
  if (st != QATTN_OK) return st;
  if (static_cast<int64_t>(batch) * view.hkv > 65535) return fail(QATTN_ERR_UNSUPPORTED, "batch * Hkv > 65535");
  if (batch == 0 || n == 0) return QATTN_OK;
  if (!k || !v) return fail(QATTN_ERR_INVALID_ARG, "k or v is NULL");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_pq_quantize(k, v, x_dtype == QATTN_F16, batch, n, start_block, view, ds->status,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "progressive quantize launch");
}

size_t qattn_decode_pq_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t max_seq_len, int32_t num_splits) {
  return qattn_decode_fp16_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_splits);
}

qattn_status qattn_decode_pq(const uint16_t *q, const qattn_pq_cache *cache, const int32_t *seq_lens, int32_t batch,
                             int32_t num_q_heads, int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                             void *workspace, size_t workspace_bytes, uint16_t *out, float *lse, qattn_stream_t stream) {
  PqView view;
  qattn_status st = check_pq(cache, &view);
  if (st != QATTN_OK) return st;
  if (batch < 0 || batch > QATTN_MAX_BATCH || num_q_heads <= 0 || max_seq_len < 0)
    return fail(QATTN_ERR_INVALID_ARG, "batch %d, Hq %d, max_seq_len %d", batch, num_q_heads, max_seq_len);
  if (num_q_heads % view.hkv) return fail(QATTN_ERR_INVALID_ARG, "Hq %d is not a multiple of Hkv %d", num_q_heads, view.hkv);
  if (num_q_heads / view.hkv > QATTN_MAX_GROUP)
    return fail(QATTN_ERR_UNSUPPORTED, "group size %d > %d", num_q_heads / view.hkv, QATTN_MAX_GROUP);
  if (num_splits < 0 || num_splits > QATTN_MAX_SPLITS)
    return fail(QATTN_ERR_INVALID_ARG, "num_splits %d (0..%d)", num_splits, QATTN_MAX_SPLITS);
  if (static_cast<int64_t>(batch) * view.hkv > 65535) return fail(QATTN_ERR_UNSUPPORTED, "batch * Hkv > 65535");
  if (batch == 0) return QATTN_OK;
  if (!q || !seq_lens || !out) return fail(QATTN_ERR_INVALID_ARG, "q, seq_lens or out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(QATTN_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  DecodePqArgs a;
  decode16_plan(batch, view.hkv, max_seq_len, num_splits, ds->sms, &a.splits, &a.chunk);
  const size_t need = decode16_workspace(batch, num_q_heads, view.head_dim, a.splits);
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return fail(QATTN_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, %zu given", need,
                workspace ? workspace_bytes : (size_t)0);
  a.q = q, a.seq_lens = seq_lens, a.out = out, a.lse = lse;
  a.partial_o = static_cast<float *>(workspace);
  const size_t rows = static_cast<size_t>(a.splits) * batch * num_q_heads;
  a.partial_lse = need ? reinterpret_cast<float *>(static_cast<char *>(workspace) + (rows * view.head_dim * 4 + 255) / 256 * 256)
                       : nullptr;
  a.batch = batch, a.hq = num_q_heads;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  cudaError_t e = launch_decode_pq(a, view, ds->status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "progressive decode launch");
}

qattn_status qattn_flashq_flush_pq(const qattn_flashq_buffer *buf, const qattn_pq_cache *cache,
                                   const int32_t *cache_lens, int32_t batch, qattn_stream_t stream) {
  FlashqView fv;
  PqView pv;
  qattn_status st = check_flashq(buf, batch, &fv);
  if (st != QATTN_OK) return st;
  if ((st = check_pq(cache, &pv)) != QATTN_OK) return st;
  if (pv.head_dim != fv.head_dim || pv.hkv != fv.hkv)
    return fail(QATTN_ERR_INVALID_ARG, "buffer (D %d, Hkv %d) and cache (D %d, Hkv %d) differ", fv.head_dim, fv.hkv,
                pv.head_dim, pv.hkv);
  if (batch == 0) return QATTN_OK;
  if (!cache_lens) return fail(QATTN_ERR_INVALID_ARG, "cache_lens is NULL");
  DeviceState *ds;
  if ((st = device_state(&ds)) != QATTN_OK) return st;
  cudaError_t e = launch_flashq_flush_pq(fv, pv, cache_lens, batch, ds->status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "flashq progressive flush launch");
}

qattn_status qattn_prefill_fp16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int32_t batch,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t capacity,
                                int32_t nq, int32_t nk, float softmax_scale, int32_t causal, uint16_t *out,
                                float *lse, qattn_stream_t stream) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || nq < 0 || nk < 0 || (causal != 0 && causal != 1))
    return fail(QATTN_ERR_INVALID_ARG, "batch %d, Hq %d, Hkv %d, nq %d, nk %d, causal %d", batch, num_q_heads,
                num_kv_heads, nq, nk, causal);
  if (num_q_heads % num_kv_heads) return fail(QATTN_ERR_INVALID_ARG, "Hq %d is not a multiple of Hkv %d", num_q_heads, num_kv_heads);
  if (head_dim != 64 && head_dim != 128) return fail(QATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (nq > nk) return fail(QATTN_ERR_INVALID_ARG, "nq %d > nk %d", nq, nk);
  if (nk > capacity || capacity > 0x7fffffffLL)
    return fail(QATTN_ERR_INVALID_ARG, "nk %d, capacity %lld", nk, (long long)capacity);
  if (batch == 0 || nq == 0) return QATTN_OK;
  if (!q || !k || !v || !out) return fail(QATTN_ERR_INVALID_ARG, "q, k, v or out is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(QATTN_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
  DeviceState *ds;
  qattn_status st = device_state(&ds);
  if (st != QATTN_OK) return st;
  CUtensorMap qmap, omap, kmap, vmap;
  if ((st = prefill_maps(&qmap, &omap, q, out, batch, num_q_heads, nq, head_dim)) != QATTN_OK) return st;
  const int64_t heads = static_cast<int64_t>(batch) * num_kv_heads;
  if ((st = fp16_cache_map(&kmap, k, heads, capacity, nk, head_dim, 128)) != QATTN_OK) return st;
  if ((st = fp16_cache_map(&vmap, v, heads, capacity, nk, head_dim, 128)) != QATTN_OK) return st;
  PrefillArgs a;
  a.q = q, a.out = out, a.lse = lse;
  a.batch = batch, a.hq = num_q_heads, a.nq = nq, a.nk = nk, a.causal = causal;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  cudaError_t e = launch_prefill16(a, num_kv_heads, head_dim, qmap, omap, kmap, vmap, ds->status,
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : cuda_fail(e, "fp16 prefill launch");
}

int32_t qattn_version(void) { return 0x000100; }

}  // extern "C"
