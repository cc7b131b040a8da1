/*
 * qattn.h -- C ABI of libqattn: attention computed directly over an INT4
 * KV cache on NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (page title and section):
 *   [QCA]   "Quantized Cross-Attention: Extending FlashAttention-3 with
 *           In-SRAM Dequantization": §3.1 in-SRAM dequantization fused into
 *           the attention loop; §3.2 tile of 4-bit codes plus one FP16 scale
 *           per token; §3.3 split-K dequantization and the 3-bit packing;
 *           §4.1 kernel signature ([batch, heads, seq, dim] ordering,
 *           compressed KV, per-token scales, output).
 *   [TA]    TurboAttention (arXiv 2412.08585): §2.1 prefill and decoding with
 *           a KV cache (K_t = K_{t-1} | k_t); §2.2 Equation 2 (S = QK^T,
 *           P = softmax(S), H = PV) and FlashAttention's tiled online
 *           softmax; §2.3 symmetric quantization (zero point 0).
 *   [OTQ]   Open-TQ-Metal abstract on the "Attention Quantization" listing:
 *           int4 KV quantized on the fly, attention on the compressed form.
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.   Every pointer is a DEVICE pointer unless marked "host".  The
 *           caller owns every buffer and the library allocates nothing.
 *           Between calls it keeps, per device that loads it, immutable
 *           kernel handles and three static device arrays: the status word
 *           of qattn_read_device_flags (4 bytes), the split scratch of
 *           qattn_decode_noalloc (QATTN_NOALLOC_SCRATCH_BYTES, 8 MiB) and
 *           the per-head statistics of qattn_headwise_plan (512 KiB).
 *           The last two are shared by every call that uses them, so such
 *           calls that overlap on the GPU race; each call rewrites every
 *           value of them it later reads.
 * Streams.  Work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *           default stream).  No call synchronises, except
 *           qattn_read_device_flags; results are ready when the stream has run.
 * Errors.   Arguments are validated on the host before any launch; a
 *           failed check returns an error code and enqueues nothing.
 *           QATTN_ERR_CUDA reports a launch failure (cudaGetLastError).
 *           qattn_last_error() gives a human-readable reason for the most
 *           recent failure on the calling thread.
 * Layout.   All tensors are dense row-major in the shapes given, 16-byte
 *           aligned.  fp16 values travel as uint16_t bit patterns.
 *
 * The KV-cache format (bit-exact; [QCA] §3.2, [TA] §2.3)
 * -------------------------------------------------------
 *   row      one (token, kv-head) vector of D values
 *   scale    s = fp16(fp32(absmax / 7)), round-to-nearest-even twice; a
 *            scale that overflows fp16 saturates to 65504
 *   codes    c_i = clamp(round_half_even(x_i / s), -7, 7) on the exact
 *            quotient; all codes 0 when s == 0
 *   packing  D/2 bytes per row; element 2k in the low nibble of byte k,
 *            element 2k+1 in the high nibble; two's complement nibbles
 *   value    x^_i = c_i * s
 *
 *   contiguous cache: codes [batch, Hkv, capacity, D/2] uint8,
 *                     scales [batch, Hkv, capacity] fp16
 *   paged cache:      codes [num_pages, Hkv, page_size, D/2] uint8,
 *                     scales [num_pages, Hkv, page_size] fp16; token t of
 *                     sequence b lives in page page_table[b*max_pages + t/page_size]
 *                     at offset t % page_size.
 *
 * Attention semantics ([TA] §2.2 Eq. 2, per head and batch instance)
 * -------------------------------------------------------------------
 *   O = softmax(softmax_scale * Q K^T + mask) V over the dequantized cache.
 *   GQA: query head h reads kv head h / (Hq / Hkv).
 *   Causal masking is bottom-right aligned: query i of Nq sees key j of Nk
 *   iff j <= i + Nk - Nq.  A decode query sees all seq_len keys.
 *   lse = natural-log log-sum-exp of the scaled scores, fp32.
 *   A query row that sees no key gives O = 0 and lse = -inf.
 */
#ifndef QATTN_H
#define QATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *qattn_stream_t;

typedef enum qattn_status {
  QATTN_OK = 0,
  QATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
  QATTN_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels cover */
  QATTN_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  QATTN_ERR_CUDA = 4         /* a CUDA runtime/driver call failed */
} qattn_status;

typedef enum qattn_dtype {
  QATTN_F32 = 0,
  QATTN_F16 = 1
} qattn_dtype;

/* Fixed limits (checked by every call). */
#define QATTN_PAGE_SIZE 64     /* tokens per page of a paged cache */
#define QATTN_MAX_GROUP 8      /* largest Hq / Hkv */
#define QATTN_MAX_SPLITS 1024  /* largest num_splits of qattn_decode */
#define QATTN_MAX_BATCH 1024   /* largest batch of qattn_decode */

/* Bits of the device status word (qattn_read_device_flags). */
#define QATTN_FLAG_WAIT_TIMEOUT 1u /* a pipeline wait gave up (kernel returned early) */
#define QATTN_FLAG_BAD_PAGE 2u     /* a page id or length was out of range; rows skipped */
#define QATTN_FLAG_TMEM 4u         /* tensor-memory allocation failed */
#define QATTN_FLAG_BUFFER_FULL 8u  /* qattn_flashq_append met a full buffer; the row was dropped */
#define QATTN_FLAG_BAD_HEAD 16u    /* a cache's kv_head_index named no head of the model; rows skipped */

/*
 * Where the quantized K and V live.  Passed by host pointer; the struct
 * itself is read during the call only.
 *   head_dim         D, 64 or 128
 *   num_kv_heads     Hkv
 *   page_table       NULL selects the contiguous layout; otherwise a device
 *                    int32 array [batch, max_pages_per_seq] of physical page
 *                    ids (-1 or any id outside [0, num_pages) = no page)
 *   capacity         contiguous layout: tokens per (sequence, kv-head);
 *                    must be a positive multiple of 64
 *   page_size        paged layout: must be QATTN_PAGE_SIZE
 *   num_pages        paged layout: pages in the pool
 *   code_bits        0 or 4: the INT4 format above.  3: INT3 ([QCA] §3.3: ten
 *                    3-bit values per little-endian 32-bit word, element j in
 *                    word j / 10 at bits 3 (j % 10), two's complement, unused
 *                    fields zero; 52 bytes per row at D = 128; scale
 *                    fp16(fp32(absmax / 3)), codes clamp(RNE(x / s), -3, 3)).
 *                    INT3 is supported by qattn_quantize_kv and qattn_decode
 *                    for a contiguous cache with D = 128; other calls return
 *                    QATTN_ERR_UNSUPPORTED for it.
 *                    2: INT2 ([TA] §3.2's 2-bit heads, read as this per-row
 *                    symmetric codec at 2 bits: sixteen 2-bit values per
 *                    little-endian 32-bit word, element j in word j / 16 at
 *                    bits 2 (j % 16), two's complement; 32 bytes per row at
 *                    D = 128; scale fp16(absmax), codes clamp(RNE(x / s),
 *                    -1, 1)).  Supported like INT3.
 *   kv_head_index    NULL: the cache holds every kv-head of the model.
 *                    Otherwise a device int32 array [num_kv_heads]: cache
 *                    head h is the model's kv-head kv_head_index[h] (one of
 *                    model_kv_heads), as in a headwise mixed-precision layout
 *                    ([TA] §3.2) that keeps the 2-bit and the 4-bit heads in
 *                    two caches.  qattn_quantize_kv then reads k, v as
 *                    [batch, model_kv_heads, n, D] and stores the listed
 *                    heads; qattn_decode attends q-heads kv_head_index[h] * G
 *                    .. + G - 1 (G = Hq / model_kv_heads) with cache head h
 *                    and writes only those rows of out and lse.  An entry
 *                    outside [0, model_kv_heads) raises QATTN_FLAG_BAD_HEAD
 *                    and its rows are skipped.  Contiguous caches only; the
 *                    other calls return QATTN_ERR_UNSUPPORTED for a listed
 *                    cache.
 *   model_kv_heads   kv-heads of the model (read when kv_head_index is set)
 */
typedef struct qattn_kv_cache {
  uint8_t *k_codes;
  uint16_t *k_scales;
  uint8_t *v_codes;
  uint16_t *v_scales;
  int32_t head_dim;
  int32_t num_kv_heads;
  const int32_t *page_table;
  int32_t max_pages_per_seq;
  int32_t page_size;
  int64_t capacity;
  int64_t num_pages;
  int32_t code_bits;
  const int32_t *kv_head_index;
  int32_t model_kv_heads;
} qattn_kv_cache;

/*
 * qattn_quantize_kv -- quantize new K and V rows and write them into the
 * cache (quantize-on-append; [TA] §2.1 K_t = K_{t-1} | k_t, codec above).
 *
 *   k, v        [batch, Hkv, n, D] of x_dtype (fp32 or fp16)
 *   batch, n    sequences, and new rows per (sequence, kv-head); n >= 0
 *   start_pos   [batch] int32: position of the first new row of each
 *               sequence; NULL means 0 for every sequence
 *   cache       destination (contiguous or paged)
 *
 * Row i of sequence b goes to token position start_pos[b] + i.  Rows whose
 * position falls at or past `capacity` (contiguous) or in a missing page
 * (paged) are not written.  Both K and V are written by one launch.
 */
qattn_status qattn_quantize_kv(const void *k, const void *v, qattn_dtype x_dtype,
                               int32_t batch, int32_t n, const int32_t *start_pos,
                               const qattn_kv_cache *cache, qattn_stream_t stream);

/*
 * qattn_decode_workspace_size -- bytes of workspace qattn_decode needs for
 * `num_splits` key ranges (0 = the automatic choice for these sizes on the
 * current device).  Host-only; returns 0 for invalid sizes.  For a cache
 * with a kv_head_index pass the model's kv-head count (model_kv_heads).
 */
size_t qattn_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_seq_len, int32_t num_splits);

/*
 * qattn_decode_plan -- the launch shape that qattn_decode and
 * qattn_decode_append (and qattn_decode_noalloc) take for these sizes on the
 * current device.  Split-KV decoding ([TA] §2.1 over [QCA] §3.3's split-K
 * partials, merged by the log-sum-exp rule of [TA] §2.2) runs one of two ways:
 *   cluster = 0   cost-balanced key ranges over `ctas` CTAs, the partials
 *                 merged by a second kernel (paged caches, listed caches,
 *                 an explicit num_splits, INT3 / INT2, or shapes whose
 *                 clusters would leave most SMs idle);
 *   cluster = S   one thread-block cluster of S CTAs (2 <= S <= 16) per
 *                 (sequence, kv-head group), ctas = batch * groups * S, the
 *                 S partials merged through distributed shared memory in the
 *                 same kernel; chosen when num_splits is 0, the cache is
 *                 contiguous INT4 without kv_head_index, every cluster can be
 *                 resident at once and the grid covers at least 80 % of the
 *                 SMs.
 *   warps  consumer warps per CTA (8: 256-row stages; 12: 384-token stages)
 *   paged  nonzero for a paged cache; code_bits 4, 3 or 2;
 *   has_kv_head_index  nonzero for a listed cache
 * The three outputs are host pointers (any may be NULL).  Host-only: reads
 * device attributes and occupancy, launches nothing.  Errors:
 * QATTN_ERR_INVALID_ARG for sizes qattn_decode would reject.
 */
qattn_status qattn_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t max_seq_len, int32_t num_splits, int32_t paged, int32_t code_bits,
                               int32_t has_kv_head_index, int32_t *warps, int32_t *ctas, int32_t *cluster);

/*
 * qattn_decode -- one query token per sequence against its whole cache
 * ([TA] §2.1 decoding; fused in-SRAM dequantization as in [QCA] §3.1).
 *
 *   q            [batch, Hq, D] fp16
 *   cache        contiguous or paged INT4 cache
 *   seq_lens     [batch] int32, 0 <= seq_lens[b] <= max_seq_len; lengths
 *                beyond the cache (capacity, or max_pages_per_seq * 64) are
 *                clamped and flagged QATTN_FLAG_BAD_PAGE
 *   max_seq_len  host int, an upper bound of seq_lens used to size the split
 *   softmax_scale multiplies Q K^T
 *   num_splits   number of balanced key ranges the whole batch is cut into
 *                (split-KV; one persistent CTA per range); 0 = one per SM.
 *                Every range holds the same number of 64-token stages, so
 *                ranges cut sequences wherever needed; a (sequence, kv-head)
 *                cut by ranges leaves one fp32 partial per range, merged by
 *                the log-sum-exp combine inside this call.
 *   workspace    device scratch of at least qattn_decode_workspace_size()
 *                bytes for the same arguments (two partial slots per range)
 *   out          [batch, Hq, D] fp16
 *   lse          [batch, Hq] fp32, or NULL
 */
qattn_status qattn_decode(const uint16_t *q, const qattn_kv_cache *cache, const int32_t *seq_lens,
                          int32_t batch, int32_t num_q_heads, int32_t max_seq_len,
                          float softmax_scale, int32_t num_splits, void *workspace,
                          size_t workspace_bytes, uint16_t *out, float *lse,
                          qattn_stream_t stream);

/*
 * qattn_decode_append -- one decoding step in one launch: each sequence's
 * new key and value rows are quantized into the cache (as qattn_quantize_kv
 * would, bit for bit) at position seq_lens[b] - 1 and attended together with
 * the cached keys ([TA] §2.1: a decoding step appends k_t, v_t to the cache,
 * then attends the new query against all of it).
 *
 *   k_new, v_new [batch, Hkv, D] of x_dtype (QATTN_F32 or QATTN_F16),
 *                16-byte aligned, read-only
 *   seq_lens     [batch] int32, lengths AFTER the append: the new row of
 *                sequence b goes to position seq_lens[b] - 1 (nothing is
 *                written for seq_lens[b] = 0); a position beyond the cache
 *                (capacity, or max_pages_per_seq * 64) is not written and is
 *                flagged QATTN_FLAG_BAD_PAGE, like a row of a missing page
 *   everything else as qattn_decode (same workspace size).
 * Errors: as qattn_decode; QATTN_ERR_INVALID_ARG for a NULL or misaligned
 * k_new / v_new or another x_dtype.
 */
qattn_status qattn_decode_append(const uint16_t *q, const void *k_new, const void *v_new, qattn_dtype x_dtype,
                                 const qattn_kv_cache *cache, const int32_t *seq_lens, int32_t batch,
                                 int32_t num_q_heads, int32_t max_seq_len, float softmax_scale,
                                 int32_t num_splits, void *workspace, size_t workspace_bytes,
                                 uint16_t *out, float *lse, qattn_stream_t stream);

/*
 * qattn_prefill -- Nq query rows per sequence against Nk cached keys
 * ([TA] §2.1 prefill, §2.2 FlashAttention tiling; dense contractions on
 * the tensor cores with the dequantization fused ahead of the operand
 * stage, [QCA] §3.1).  Contiguous or paged cache (chunked prefill of a
 * paged cache: the new rows' Q against every cached key).
 *
 *   q        [batch, Hq, Nq, D] fp16
 *   nq, nk   query rows and keys per sequence, 1 <= nq <= nk <= capacity
 *            (paged: nk <= max_pages_per_seq * 64; a key in a missing page
 *            raises QATTN_FLAG_BAD_PAGE and leaves that sequence's rows
 *            undefined)
 *   causal   0 or 1 (bottom-right aligned)
 *   out      [batch, Hq, Nq, D] fp16
 *   lse      [batch, Hq, Nq] fp32, or NULL
 */
qattn_status qattn_prefill(const uint16_t *q, const qattn_kv_cache *cache, int32_t batch,
                           int32_t num_q_heads, int32_t nq, int32_t nk, float softmax_scale,
                           int32_t causal, uint16_t *out, float *lse, qattn_stream_t stream);

/*
 * qattn_combine -- log-sum-exp merge of split-KV partial results ([TA]
 * §2.2: FlashAttention's online softmax keeps a running max and sum per
 * row, so two partial results over disjoint key sets merge exactly by
 * rescaling each with exp(lse_c - L); [QCA] §3.3 splits the key dimension
 * across thread blocks and needs this merge).
 *
 *   partial_o    [num_splits, rows, D] fp32, each normalised within its split
 *   partial_lse  [num_splits, rows] fp32 (natural log); a split with
 *                lse = -inf saw no key and its partial_o is never read
 *   out          [rows, D] fp16:  O = sum_c exp(lse_c - L) O_c,
 *   lse          [rows] fp32 or NULL:  L = ln sum_c exp(lse_c)
 * Rows whose every split is empty get O = 0 and lse = -inf.
 */
qattn_status qattn_combine(const float *partial_o, const float *partial_lse, int32_t num_splits,
                           int64_t rows, int32_t head_dim, uint16_t *out, float *lse,
                           qattn_stream_t stream);

/*
 * qattn_read_device_flags -- synchronise the current device, return in
 * *flags (host) the OR of QATTN_FLAG_* bits the kernels raised since the
 * last clear, and clear them if `clear` is non-zero.
 */
qattn_status qattn_read_device_flags(uint32_t *flags, int32_t clear);

/*
 * qattn_check_wait_timeout -- exercises the bounded waits every kernel of
 * the library uses, without faulting or hanging the GPU.  One small kernel
 * waits on an mbarrier that no thread ever arrives at, gives up after
 * `limit_cycles` SM clock cycles (1 ... 2^31), and writes the QATTN_FLAG_*
 * bits it raised to *flags (device, uint32): QATTN_FLAG_WAIT_TIMEOUT when
 * the wait gave up as it must.  The device status word of
 * qattn_read_device_flags is not touched and the context stays usable.  The
 * pages have no counterpart: this is the library's own failure check.
 */
qattn_status qattn_check_wait_timeout(uint32_t *flags, int64_t limit_cycles, qattn_stream_t stream);

/*
 * FlashQ-style decode buffer ([TA] §3.3): decoded K/V rows wait in a buffer
 * of QATTN_FLASHQ_ROWS rows per (sequence, kv-head) as int8 codes with one
 * universal scale per (sequence, kv-head) and tensor, outliers clamped, and
 * a full buffer is compressed into the INT4 cache.  Readings of the page
 * (which gives no formula for the universal scale):
 *   R      running max |x^| of the rows already cached for that (sequence,
 *          kv-head) and tensor = 7 * their largest INT4 scale; while R is 0
 *          (no or all-zero history) each appended row sets R to its absmax
 *   u      fp16(fp32(R / 127)), both roundings to nearest even, saturating
 *   code   clamp(round_half_even(x / u), -127, 127) on the exact quotient
 *   value  x~ = code * u
 *   flush  a full buffer's x~ rows go through the INT4 codec into the cache
 *          at positions cache_lens[b] .. cache_lens[b] + 63; R rises to the
 *          new rows' 7 * max scale if larger; u follows; the buffer empties
 * A decode step with the buffer: qattn_decode over the cached rows (with an
 * lse array), qattn_flashq_append of the step's new rows, qattn_flashq_attend
 * (merges the buffered rows into out / lse), and every 64 steps
 * qattn_flashq_flush (then the caller's cached lengths grow by 64).
 * Sequences advance together: one appended row per sequence per call.
 */
#define QATTN_FLASHQ_ROWS 64

typedef struct qattn_flashq_buffer {
  int8_t *k_codes;     /* [batch, Hkv, 64, D] int8, 16-byte aligned */
  int8_t *v_codes;     /* [batch, Hkv, 64, D] int8, 16-byte aligned */
  uint16_t *k_scale;   /* [batch, Hkv] fp16 universal scales u */
  uint16_t *v_scale;   /* [batch, Hkv] fp16 */
  float *k_range;      /* [batch, Hkv] R */
  float *v_range;      /* [batch, Hkv] R */
  int32_t *count;      /* [batch] rows buffered, 0..64 */
  int32_t head_dim;    /* D: 64 or 128, as the cache */
  int32_t num_kv_heads; /* Hkv (1..64), as the cache */
} qattn_flashq_buffer;

/* R and u from the first cache_lens[b] cached rows of every (sequence,
 * kv-head); empties the buffers.  cache_lens: device int32 [batch]. */
qattn_status qattn_flashq_init(const qattn_flashq_buffer *buf, const qattn_kv_cache *cache,
                               const int32_t *cache_lens, int32_t batch, qattn_stream_t stream);

/* One new K and V row per (sequence, kv-head): k_new, v_new [batch, Hkv, D]
 * of x_dtype (QATTN_F32 or QATTN_F16), 16-byte aligned.  A full buffer drops
 * the row and raises QATTN_FLAG_BUFFER_FULL. */
qattn_status qattn_flashq_append(const void *k_new, const void *v_new, qattn_dtype x_dtype,
                                 const qattn_flashq_buffer *buf, int32_t batch, qattn_stream_t stream);

/* Merges attention over the buffered rows into out [batch, Hq, D] fp16 and
 * lse [batch, Hq] fp32 (required), which hold a decode over the cached rows
 * (lse = -inf where those were empty): L = log(e^lse + e^lse_buf), out =
 * e^(lse - L) out + e^(lse_buf - L) O_buf.  q [batch, Hq, D] fp16, the same
 * query; GQA as in qattn_decode.  Sequences with an empty buffer are left as
 * they are.  The buffered rows are attended while the preceding decode on the
 * stream may still run (a programmatic launch; out and lse are read after
 * it completes), so q must not be that decode's out. */
qattn_status qattn_flashq_attend(const uint16_t *q, const qattn_flashq_buffer *buf, int32_t batch,
                                 int32_t num_q_heads, float softmax_scale, uint16_t *out, float *lse,
                                 qattn_stream_t stream);

/* Moves every full buffer into the cache at positions cache_lens[b] ..
 * cache_lens[b] + 63 (device int32 [batch], the rows already cached); rows
 * past the cache or in a missing page are not written and raise
 * QATTN_FLAG_BAD_PAGE.  Buffers that are not full are untouched. */
qattn_status qattn_flashq_flush(const qattn_flashq_buffer *buf, const qattn_kv_cache *cache,
                                const int32_t *cache_lens, int32_t batch, qattn_stream_t stream);

/* Bytes of the library-owned scratch behind qattn_decode_noalloc (8 MiB per device). */
#define QATTN_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * qattn_decode_noalloc -- qattn_decode without a workspace argument, for
 * callers that cannot allocate device memory (for example a plugin that is
 * handed only its input and output buffers, or code on a device whose memory
 * a caching allocator has already reserved).  The source pages have no
 * counterpart; this is a convenience of the library.
 *
 * Same arguments and results as qattn_decode, except that the split partials
 * live in a fixed device array owned by the library
 * (QATTN_NOALLOC_SCRATCH_BYTES on every GPU that loads it, kept until exit).
 *   - Sizes whose partials exceed that array are refused with
 *     QATTN_ERR_UNSUPPORTED before any work (use fewer splits, or qattn_decode).
 *   - The first call on a device, with that device current, looks up the
 *     array's address (cudaGetSymbolAddress); make it before any stream capture.
 *   - All calls on a device share the array: calls that overlap on the GPU
 *     race.  Nothing in it needs clearing between calls.
 *   - The call allocates nothing.
 */
qattn_status qattn_decode_noalloc(const uint16_t *q, const qattn_kv_cache *cache,
                                  const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                  int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                                  uint16_t *out, float *lse, qattn_stream_t stream);

/*
 * qattn_headwise_plan -- the headwise mixed-precision plan of [TA] §3.2:
 * one priority per kv-head from a prompt's keys and values, and 2 bits for
 * the num_low heads of lowest priority, 4 bits for the others.
 *
 *   k, v       [batch, Hkv, n, D] of x_dtype (fp32 or fp16), finite values;
 *              the layout qattn_quantize_kv reads
 *   lens       [batch] int32 (device) rows of each sequence that count
 *              (clamped to [0, n]); NULL = all n
 *   num_low    n_h, 0 <= num_low <= Hkv
 *   bits       [Hkv] int32 (device), written: 2 or 4
 *   priority   [Hkv] float64 (device), written when not NULL
 *
 * The page names the two statistics and omits the equation that combines
 * them; this library's reading: per head and tensor, with mx_j and mn_j the
 * largest and smallest value of channel j over the counted rows,
 * gap = max_j mx_j - min_j mn_j, std = the population standard deviation of
 * the channel gaps mx_j - mn_j, priority = gap * std; a kv-head's priority
 * is the larger of its key and value priorities (its K and V share one bit
 * width); ties go to the lower head index.  The statistics are binary64,
 * summed in channel order without fused multiply-adds, so they are
 * reproducible bit for bit.  Hkv <= 256.  Calls that overlap on the GPU
 * race (they share one device scratch array).
 */
qattn_status qattn_headwise_plan(const void *k, const void *v, qattn_dtype x_dtype, int32_t batch,
                                 int32_t num_kv_heads, int32_t n, int32_t head_dim, const int32_t *lens,
                                 int32_t num_low, int32_t *bits, double *priority, qattn_stream_t stream);

/*
 * Comparison paths ([QCA] §5.2 Baselines, §5.3 Results): the page measures
 * the fused 4-bit kernel against an FP16 FlashAttention kernel over an FP16
 * KV cache, and against "post-dequantization", where the 4-bit cache is
 * first written back to HBM in FP16 and then attended.  These calls build
 * both arms on this GPU, so that what fusion saves can be measured here.
 * They follow the conventions above (GQA, bottom-right causal, lse, empty
 * rows); an FP16 cache is K, V [batch, Hkv, capacity, D] fp16, contiguous.
 */

/*
 * qattn_dequantize_kv -- the first n tokens of every (sequence, kv-head) of
 * an INT4 cache (contiguous or paged) written out as fp16:
 *   k_out, v_out  [batch, Hkv, n, D] fp16, x16 = fl16(c * s) (the exact
 *                 product rounded once to binary16, ties to even; products
 *                 beyond the fp16 range become +-inf)
 * n must not exceed the cache (capacity, or max_pages_per_seq * 64); a token
 * in a missing page is written as zeros and raises QATTN_FLAG_BAD_PAGE.
 * INT4 caches without kv_head_index only (QATTN_ERR_UNSUPPORTED otherwise).
 */
qattn_status qattn_dequantize_kv(const qattn_kv_cache *cache, int32_t batch, int32_t n, uint16_t *k_out,
                                 uint16_t *v_out, qattn_stream_t stream);

/* Workspace bytes of qattn_decode_fp16 for these sizes (0 when one key range
 * suffices, and for invalid sizes).  Host-only. */
size_t qattn_decode_fp16_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_seq_len, int32_t num_splits);

/*
 * qattn_decode_fp16 -- qattn_decode over an FP16 cache.
 *   q          [batch, Hq, D] fp16
 *   k, v       [batch, Hkv, capacity, D] fp16 (capacity >= max_seq_len)
 *   seq_lens   [batch] int32 (device), clamped to [0, capacity]
 *   num_splits key ranges per (sequence, kv-head), 0 = one CTA per SM in all;
 *              each range is a multiple of 64 tokens; with more than one the
 *              partials are merged as qattn_combine does
 *   workspace  qattn_decode_fp16_workspace_size() bytes (may be 0 / NULL)
 *   out, lse   [batch, Hq, D] fp16, [batch, Hq] fp32 or NULL
 * batch * Hkv <= 65535.
 */
qattn_status qattn_decode_fp16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int32_t batch,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t capacity,
                               const int32_t *seq_lens, int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                               void *workspace, size_t workspace_bytes, uint16_t *out, float *lse,
                               qattn_stream_t stream);

/*
 * qattn_prefill_fp16 -- qattn_prefill over an FP16 cache: q [batch, Hq, Nq, D]
 * against the first nk keys of k, v [batch, Hkv, capacity, D] fp16,
 * 1 <= nq <= nk <= capacity; out [batch, Hq, Nq, D] fp16, lse [batch, Hq,
 * Nq] fp32 or NULL.  The same tensor-core kernel as qattn_prefill, with K
 * and V tiles loaded by TMA instead of dequantized.
 */
qattn_status qattn_prefill_fp16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int32_t batch,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t capacity,
                                int32_t nq, int32_t nk, float softmax_scale, int32_t causal, uint16_t *out,
                                float *lse, qattn_stream_t stream);

/*
 * Progressive INT8 -> INT4 storage ([TA] §3.1 Blockwise Progressive
 * Quantization; §3.3 compresses a full decode buffer this way).  The cache is
 * kept in blocks of 64 tokens of one (sequence, kv-head) and tensor; the page
 * gives no equations, and this library's reading is (every step exact):
 *   s1  = fp16(fp32(absmax(block) / 127)), round-to-nearest-even twice,
 *         saturating; q1 = clamp(RNE(x / s1), -127, 127), 0 when s1 == 0
 *   per channel d of the block: lo = min q1, hi = max q1,
 *   s2  = max(1, ceil((hi - lo) / 15)), z2 = lo,
 *   q2  = RNE((q1 - lo) / s2) on the exact rational, 0..15
 *   value x^ = (q2 * s2 + z2) * s1
 *
 *   k_codes, v_codes    [batch, Hkv, capacity, D/2] uint8: q2 as unsigned
 *                       nibbles, element 2k in the low nibble of byte k
 *   k_params, v_params  [batch, Hkv, capacity/64, 2*D + 16] uint8, one record
 *                       per block: s2[D] (uint8), z2[D] (int8), s1 (fp16), 14
 *                       zero bytes
 *   capacity            tokens per (sequence, kv-head), a multiple of 64
 * All four pointers 16-byte aligned.  D = 64 or 128.
 */
typedef struct qattn_pq_cache {
  uint8_t *k_codes;
  uint8_t *v_codes;
  uint8_t *k_params;
  uint8_t *v_params;
  int32_t head_dim;
  int32_t num_kv_heads;
  int64_t capacity;
} qattn_pq_cache;

/*
 * qattn_pq_quantize -- n new rows per (sequence, kv-head), n a multiple of
 * 64, k and v [batch, Hkv, n, D] of x_dtype (fp32 or fp16), stored as n / 64
 * blocks at block positions start_block[b] + i (device int32 [batch]; NULL
 * means 0).  A block past the cache is not written and raises
 * QATTN_FLAG_BAD_PAGE.  batch * Hkv <= 65535.
 */
qattn_status qattn_pq_quantize(const void *k, const void *v, qattn_dtype x_dtype, int32_t batch, int32_t n,
                               const int32_t *start_block, const qattn_pq_cache *cache, qattn_stream_t stream);

/* Workspace bytes of qattn_decode_pq (the same key ranges as qattn_decode_fp16). */
size_t qattn_decode_pq_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t max_seq_len, int32_t num_splits);

/*
 * qattn_decode_pq -- qattn_decode over a progressive cache: q [batch, Hq,
 * D] fp16, seq_lens [batch] int32 (device; whole blocks: a length that is
 * not a multiple of 64 attends the block's leading tokens only), key ranges
 * and workspace as qattn_decode_fp16, out [batch, Hq, D] fp16, lse [batch,
 * Hq] fp32 or NULL.  Each block is dequantized on chip (INT4 -> the exact
 * integer q1' in fp16 -> the MMA, s1 applied to the scores and to P); no
 * fp16 copy of K or V is written to HBM.
 */
qattn_status qattn_decode_pq(const uint16_t *q, const qattn_pq_cache *cache, const int32_t *seq_lens, int32_t batch,
                             int32_t num_q_heads, int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                             void *workspace, size_t workspace_bytes, uint16_t *out, float *lse, qattn_stream_t stream);

/*
 * qattn_flashq_flush_pq -- a full decode buffer ([TA] §3.3: once it holds 64
 * rows it is compressed by progressive quantization) into one block of a
 * progressive cache: its int8 codes are stage 1 already (s1 = the buffer's
 * universal scale u), stage 2 runs on them, and the block goes to token
 * position cache_lens[b] (device int32 [batch], a multiple of 64; otherwise,
 * or past the cache, nothing is written and QATTN_FLAG_BAD_PAGE is raised).
 * The buffer empties; its range R and scale u are kept (the universal range
 * already bounds the block).  Buffers that are not full are untouched.  The
 * buffer and the cache must have the same D and Hkv.
 */
qattn_status qattn_flashq_flush_pq(const qattn_flashq_buffer *buf, const qattn_pq_cache *cache,
                                   const int32_t *cache_lens, int32_t batch, qattn_stream_t stream);

/* Static description of a status code (never NULL). */
const char *qattn_status_string(qattn_status status);

/* Reason for the most recent non-OK status on the calling thread (host). */
const char *qattn_last_error(void);

/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t qattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QATTN_H */
