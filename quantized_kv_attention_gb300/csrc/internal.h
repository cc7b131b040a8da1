// internal.h -- launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qattn {

// Device view of a KV cache (contiguous or paged), passed by value to kernels.
struct KvView {
  uint8_t *k_codes;
  uint16_t *k_scales;
  uint8_t *v_codes;
  uint16_t *v_scales;
  const int32_t *page_table;  // nullptr = contiguous
  int64_t capacity;           // contiguous: tokens per (sequence, kv-head)
  int64_t num_pages;          // paged: pool size
  int32_t max_pages;          // paged: page-table row length
  int32_t hkv;
  int32_t head_dim;
  int32_t bits;               // 4 (INT4), 3 (INT3) or 2 (INT2); INT3 and INT2: contiguous, D = 128
  // A cache holding some of a model's kv-heads: cache head h is the model's
  // kv-head head_map[h] of model_hkv (nullptr: h itself, model_hkv = hkv).
  const int32_t *head_map;
  int32_t model_hkv;
};

constexpr int kPage = 64;  // tokens per page and per decode pipeline stage

// Status bit QATTN_FLAG_BAD_HEAD: a cache's head map named no head of the
// model (its rows were skipped).
constexpr uint32_t kFlagBadHead = 16u;

// The model's kv-head of cache head h (KvView::head_map); -1 when the map
// names no head of the model.
__device__ __forceinline__ int model_head(const int32_t *head_map, int model_hkv, int h) {
  if (!head_map) return h;
  const int m = __ldg(head_map + h);
  return m >= 0 && m < model_hkv ? m : -1;
}

// quantize.cu
// (a persistent grid of four CTAs per SM: `sms` = the device's SM count)
cudaError_t launch_quantize(const void *k, const void *v, bool fp16_in, int batch, int n,
                            const int32_t *start_pos, const KvView &cache, uint32_t *err, int sms,
                            cudaStream_t stream);

// decode.cu: persistent split-KV decode over `ctas` balanced key ranges plus
// the merge of segments the ranges cut.  A stage carries 256 (token, kv-head)
// rows: tokens_per_stage tokens of heads_per_stage kv-heads.  Workspace:
// partial_o [2*ctas, heads_per_stage*G, D] and partial_lse [2*ctas,
// heads_per_stage*G] fp32 (two slots per CTA).
struct DecodeArgs {
  const uint16_t *q;
  const int32_t *seq_lens;
  uint16_t *out;
  float *lse;
  float *partial_o;
  float *partial_lse;
  // fused append: the new K and V rows [batch, Hkv, D] (fp32, or fp16 when
  // new_fp16), quantized into the cache at position seq_lens[b] - 1 before
  // they are attended; NULL for a plain decode
  const void *k_new, *v_new;
  int new_fp16;
  int max_len;       // the caller's bound of seq_lens (a guess for early prefetches)
  int batch, hq, ctas;
  int warps;         // CTA layout: 8 or 12 consumer warps (decode_layout)
  float scale_log2;  // softmax_scale * log2(e)
  int auto_splits;   // the caller left the split count to the library
  int sms;           // SM count of the device
  int cluster;       // set by launch_decode: CTAs per segment cluster (0: cost-balanced ranges + merge kernel)
};
struct DecodeGeometry {
  int heads_per_stage, tokens_per_stage, groups;
  int box_heads, box_tokens, box_rows;  // TMA boxes of codes (rows of 128 B) and scales
};
// CTA layout of a decode call: 12 consumer warps on 384-token stages for a
// contiguous cache with at least 12 such stages of work per range (long
// sequences), else 8 warps on 256-row stages.  `ranges` = the requested
// split count, or the SM count for the automatic choice.
int decode_layout(int batch, int hkv, int max_len, bool paged, int ranges);
DecodeGeometry decode_geometry(int head_dim, int hkv, bool paged, int warps);
// Segment-cluster size of a decode launch (0: cost-balanced ranges and the
// merge kernel); see launch_decode.  Host-only.
int decode_cluster(int head_dim, int warps, int bits, bool auto_splits, bool paged, bool head_map, int batch,
                   int hkv, int64_t max_len, int sms);
struct DecodeMaps {
  CUtensorMap k, v, ks, vs;  // codes 3-D [heads][rows][128 B], scales 2-D [heads][tokens]
};
// The decode buffer of qattn_flashq_* (see include/qattn.h).
struct FlashqView {
  int8_t *k_codes, *v_codes;    // [batch, Hkv, 64, D] int8 codes
  uint16_t *k_scale, *v_scale;  // [batch, Hkv] fp16 universal scales
  float *k_range, *v_range;     // [batch, Hkv] running max |x^| of the cached rows
  int32_t *count;               // [batch] rows buffered
  int hkv, head_dim;
};
cudaError_t launch_flashq_init(const FlashqView &f, const KvView &c, const int32_t *cache_lens, int batch,
                               cudaStream_t stream);
cudaError_t launch_flashq_append(const void *k, const void *v, bool fp16_in, const FlashqView &f, int batch,
                                 uint32_t *err, cudaStream_t stream);
cudaError_t launch_flashq_attend(const uint16_t *q, const FlashqView &f, int batch, int hq, float scale_log2,
                                 uint16_t *out, float *lse, cudaStream_t stream);
cudaError_t launch_flashq_flush(const FlashqView &f, const KvView &c, const int32_t *cache_lens, int batch,
                                uint32_t *err, cudaStream_t stream);

cudaError_t launch_decode(const DecodeArgs &a, const KvView &cache, const DecodeMaps &maps, uint32_t *err,
                          cudaStream_t stream);

// headwise.cu: priorities of the kv-heads of k, v [batch, Hkv, n, D] and
// bits[h] = 2 for the n_low lowest, else 4 (see include/qattn.h).
int headwise_max_heads();
cudaError_t launch_headwise_plan(const void *k, const void *v, bool fp16_in, int batch, int hkv, int n,
                                 int head_dim, const int32_t *lens, int n_low, int32_t *bits, double *priority,
                                 cudaStream_t stream);

// combine.cu (pdl: launched as a programmatic dependent of the previous kernel)
cudaError_t launch_combine(const float *partial_o, const float *partial_lse, int splits,
                           int64_t rows, int head_dim, uint16_t *out, float *lse, bool pdl,
                           cudaStream_t stream);

// prefill.cu
struct PrefillArgs {
  const uint16_t *q;
  uint16_t *out;
  float *lse;
  int batch, hq, nq, nk, causal;
  float scale_log2;
};
// qmap / omap: 3-D [batch*Hq][nq][D] fp16, 128B swizzle, boxes of 64 columns
// x 128 rows (Q) and x 32 rows (O).
cudaError_t launch_prefill(const PrefillArgs &a, const KvView &cache, const CUtensorMap &qmap,
                           const CUtensorMap &omap, uint32_t *err, cudaStream_t stream);
// prefill over an fp16 cache (comparison path): kmap / vmap 3-D
// [batch*Hkv][nk][D] fp16, 128B swizzle, boxes of 64 columns x 128 keys.
cudaError_t launch_prefill16(const PrefillArgs &a, int hkv, int head_dim, const CUtensorMap &qmap,
                             const CUtensorMap &omap, const CUtensorMap &kmap, const CUtensorMap &vmap, uint32_t *err,
                             cudaStream_t stream);

// fp16kv.cu: the comparison paths.  dequantize: the first n tokens of every
// (sequence, kv-head) of an INT4 cache -> fp16 [batch, Hkv, n, D] (K and V).
cudaError_t launch_dequantize(const KvView &cache, int batch, int n, uint16_t *k_out, uint16_t *v_out, uint32_t *err,
                              int sms, cudaStream_t stream);
// decode over an fp16 cache [batch, Hkv, capacity, D] (kmap, vmap: 3-D
// [batch*Hkv][capacity][D], 128B swizzle, boxes of 64 columns x 64 tokens);
// `splits` key ranges of `chunk` tokens; partials [splits, batch*Hq, D] and
// [splits, batch*Hq] fp32 when splits > 1, merged by the combine kernel.
struct Decode16Args {
  const uint16_t *q;
  const int32_t *seq_lens;
  uint16_t *out;
  float *lse;
  float *partial_o, *partial_lse;
  int batch, hq, hkv, head_dim, splits, chunk;
  int64_t capacity;
  float scale_log2;
};
cudaError_t launch_decode16(const Decode16Args &a, const CUtensorMap &kmap, const CUtensorMap &vmap, uint32_t *err,
                            cudaStream_t stream);

// pq.cu: progressive INT8 -> INT4 storage in 64-token blocks.  Codes [batch,
// Hkv, capacity, D/2] unsigned nibbles; one record per (sequence, kv-head,
// block) and tensor [batch, Hkv, capacity/64, 2*D + 16] bytes: s2[D] uint8,
// z2[D] int8, s1 fp16, 14 zero bytes.
struct PqView {
  uint8_t *k_codes, *v_codes;
  uint8_t *k_params, *v_params;
  int64_t capacity;
  int hkv, head_dim;
};
// n new tokens per (sequence, kv-head), a multiple of 64, into blocks
// start_block[b] + i (start_block NULL: 0); blocks past the cache are skipped.
cudaError_t launch_pq_quantize(const void *k, const void *v, bool fp16_in, int batch, int n, const int32_t *start_block,
                               const PqView &c, uint32_t *err, cudaStream_t stream);
// decode over a progressive cache: `splits` key ranges of `chunk` tokens (a
// multiple of 64); partials as Decode16Args.
struct DecodePqArgs {
  const uint16_t *q;
  const int32_t *seq_lens;
  uint16_t *out;
  float *lse;
  float *partial_o, *partial_lse;
  int batch, hq, splits, chunk;
  float scale_log2;
};
cudaError_t launch_decode_pq(const DecodePqArgs &a, const PqView &c, uint32_t *err, cudaStream_t stream);
// full decode buffers -> one progressive block each at cache_lens[b]
cudaError_t launch_flashq_flush_pq(const FlashqView &f, const PqView &c, const int32_t *cache_lens, int batch,
                                   uint32_t *err, cudaStream_t stream);

// api.cu: sets the message returned by qattn_last_error() on this thread.
void record_error(const char *msg);

}  // namespace qattn
