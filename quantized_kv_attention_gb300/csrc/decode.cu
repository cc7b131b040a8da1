// decode.cu -- split-KV decode attention over the INT4 (INT3, INT2) cache.
//
// TurboAttention (arXiv 2412.08585) §2.1: a decode step attends the new query
// q_t against the whole cache; §2.2: FlashAttention's tiling with the online
// softmax of Milakov & Gimelshein (running max and sum, rescaling, final
// normalisation), here split along the keys with a log-sum-exp merge.
// "Quantized Cross-Attention ... In-SRAM Dequantization" §3.1-§3.2: the 4-bit
// tile goes from HBM into shared memory and is dequantized inline, never
// written back as fp16; a quantized tile is 4x smaller, so a deep ring of
// tiles fits on chip.
//
// Stage.  One pipeline stage holds 32 (token, kv-head) rows per consumer
// warp: 256 rows with 8 consumer warps (a contiguous cache: 256 tokens of one
// kv-head; a paged pool: one 64-token page of 4 kv-heads, or 256/Hkv tokens of
// every head when Hkv < 4), 384 tokens of one kv-head with 12 consumer warps
// (contiguous caches whose ranges hold at least 12 such stages).  It arrives
// as a few large TMA requests -- K codes, V codes (16 or 24 KB at D = 128), K
// scales, V scales: few large requests are what lets one CTA per SM stream at
// HBM speed.
//
// Work split.  Stages of all (sequence, head-group) segments form one list;
// a persistent grid of one CTA per SM cuts it into contiguous ranges of equal
// cost (a stage, plus a fixed share for each segment a range starts), so every
// SM does the same work whatever the lengths.  A
// segment inside one range is finished by its CTA (fp16 O and lse); a segment
// cut by range boundaries leaves one fp32 partial per CTA it touches, merged
// by decode_merge_kernel (launched as a programmatic dependent, small enough
// to be resident beside the decode CTAs).
//
// Segment clusters.  When the split count is left to the library and the
// cache is contiguous INT4 without a head map, every segment may instead get
// a thread-block cluster of S CTAs (S = min(16, SMs / segments, stages); kept
// only if all clusters fit at once and cover at least 80 % of the SMs): CTA
// rank r takes the segment's stages [r n / S, (r + 1) n / S), leaves its
// normalised partial in its own Q slot, and after a cluster barrier the CTAs
// merge the S partials through distributed shared memory, each a share of the
// output columns -- no merge kernel, no partials in global memory, and the
// next call's CTAs can start as soon as SMs free up (decode_kernel<..., true>).
//
// CTA roles (W = 8 or 12 consumer warps).
//   producer    one elected thread of warp W issues the stage's TMA loads
//               into a 6-deep (W = 8) or 4-deep (W = 12) mbarrier ring; with
//               W = 12 warps W..W+3 form a warpgroup that hands its registers
//               to the consumers (setmaxnreg).
//   warps 0..W-1 consumers: warp w owns kv-head w / (W / HB) of the stage and
//               32 tokens of it (HB = kv-heads per stage).
//     S^T (16 tokens x 8 q-heads) = codes_K . Q^T on mma.sync m16n8k16 with
//       tokens on M.  A nibble becomes the fp16 subnormal u * 2^-24,
//       u = code + 8, in one LOP3 (a high nibble gives 16 u * 2^-24 and Q
//       carries 1/16 for those columns); S = 2^24 acc - 8 sum(q), exact.
//     online softmax in the log2 domain, K scale per token in fp32, one max
//       reduction per 32 tokens, warp-uniform rescale when the max grows.
//     P' = P * s_V[token] in fp16, moved to the B-operand layout by movmatrix.
//     O^T (D x 8 q-heads) += V codes^T . P'^T, V transposed by ldmatrix.trans
//       and decoded the same way; O = 2^24 / f acc - 8 sum(P').
//   INT3 and INT2 rows take the same path with their own field extraction
//   (ext3, decode_sub2), code offsets 4 and 2, and Q columns scaled to match.
//   A cache listing some of a model's kv-heads (head_map) reads the Q rows and
//   writes the output rows of the model head each of its heads stands for.
#include <math.h>

#include "../../include/qattn.h"
#include "internal.h"
#include "ptx.cuh"
#include "quant_row.cuh"

namespace qattn {
namespace {

constexpr float kTwo24 = 16777216.0f;

// Two CTA layouts, by the number W of consumer warps (32 tokens each per
// stage):
//   W = 8   stages of 256 rows, one producer warp, 9 warps (paged pools: a
//           stage is one 64-token page of 4 kv-heads)
//   W = 12  stages of 384 tokens of one kv-head (contiguous caches), three
//           consumer warps per SM sub-partition; a producer warpgroup whose
//           registers go to the consumers (setmaxnreg: 3 x 160 + 32 = 4 x 128)
// Largest segment cluster (CTAs that share one segment and merge through
// distributed shared memory): 16, a non-portable cluster size.
constexpr int kMaxCluster = 16;

template <int W>
struct Layout {
  static constexpr int kConsumerWarps = W;
  static constexpr int kRows = 32 * W;  // (token, kv-head) rows per stage
  static constexpr bool kSplitRegs = W > 8;
  static constexpr int kThreads = kSplitRegs ? (W + 4) * 32 : (W + 1) * 32;
  static constexpr int kRegsConsumer = 160, kRegsProducer = 32;
};

// BITS = 4: the INT4 rows (D/2 bytes); BITS = 3: INT3 rows of ten 3-bit
// values per 32-bit word (D = 128: 13 words, 52 bytes), read unswizzled;
// BITS = 2: INT2 rows of sixteen 2-bit values per word (D = 128: 32 bytes).
template <int D, int W, int BITS = 4>
struct Cfg {
  static constexpr int kRows = Layout<W>::kRows;
  static constexpr int kTokBytes = BITS == 3 ? 52 : BITS == 2 ? D / 4 : D / 2;  // code bytes per (token, kv-head)
  static constexpr int kCodeBytes = kRows * kTokBytes;      // per tensor per stage
  static constexpr int kScaleBytes = kRows * 2;
  // the last stage of a segment also hosts the cross-warp merge area
  static constexpr int kDataBytes = (2 * kCodeBytes + 2 * kScaleBytes + 1023) / 1024 * 1024;
  static constexpr int kMergeBytes = (W * 8 * (D + 4) * 4 + 1023) / 1024 * 1024;
  static constexpr int kStageBytes = kDataBytes > kMergeBytes ? kDataBytes : kMergeBytes;
  static constexpr int kStages = D == 128 ? (W == 8 ? 6 : 4) : (W == 8 ? 12 : 8);
  static constexpr int kQSlot = 4 * QATTN_MAX_GROUP * D * 2;  // Q rows of one segment (<= 4 kv-heads)
  // fp32 row pitch of the cross-warp merge area laid over the last stage's
  // buffer ([W warps][8 q-heads][pitch]); with 4 words of padding the eight
  // float4 stores of one quarter-warp (rows 2c, d = 4g) start 8c + 4g words
  // apart modulo 32 banks, so they never share a bank
  static constexpr int kMergePitch = D + 4;
  static_assert(W * 8 * kMergePitch * 4 <= kStageBytes, "merge area fits a stage");
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kKBytes = kTokBytes / 4;  // K code bytes per lane per token (INT4, INT2)
  static constexpr int kWords = kKBytes / 4;
  static constexpr int kMt = D / 16;     // m-tiles of O^T, k-steps of S
  // INT3: k-steps of S (10 words' pairs per lane), m-tiles of O^T (5 pairs of
  // each of a lane's 2 words)
  static constexpr int kKs3 = 10, kMt3 = 10;
  static constexpr int kOt = BITS == 3 ? kMt3 : kMt;
};

// Dynamic shared memory: ring | Q slot | m, l per (warp, q-head) | prefix |
// lengths | non-empty prefix | barriers, flags.  The cross-warp merge reuses a
// ring slot.
template <int D, int W, int BITS = 4>
__host__ __device__ constexpr int smem_bytes(int batch) {
  return Cfg<D, W, BITS>::kRing + Cfg<D, W, BITS>::kQSlot + 2 * W * 8 * 4 + (3 * batch + 2) * 4 +
         (2 * Cfg<D, W, BITS>::kStages + 3) * 8 + Cfg<D, W, BITS>::kStages * 4 + 32 + 1024;
}

template <int W>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory");
}

// Nibbles -> fp16 subnormals: out[k] = (u_lo, u_hi) * 2^-24 for nibble k of
// each 16-bit half, u = code + 8 (the XOR maps two's complement to offset
// binary); odd k come out 16x larger (the nibble sits four bits higher).
__device__ __forceinline__ void decode_sub(uint32_t w, uint32_t (&out)[4]) {
  const uint32_t w8 = w >> 8;
  out[0] = lop3_and_xor(w, 0x000F000Fu, 0x00080008u);
  out[1] = lop3_and_xor(w, 0x00F000F0u, 0x00800080u);
  out[2] = lop3_and_xor(w8, 0x000F000Fu, 0x00080008u);
  out[3] = lop3_and_xor(w8, 0x00F000F0u, 0x00800080u);
}

// INT2 word -> eight MMA registers of fp16 subnormals: out[e] = (field e,
// field e + 8) * 4^(e & 3) * 2^-24 as u = code + 2 (the XOR flips each
// 2-bit field's sign bit); fields 4..7 of each half are read after a shift
// by 8, so no field reaches the exponent bits.  For a K word the two fields
// are elements e and e + 8 of one row; for an ldmatrix.trans word of V they
// are element e of two tokens.
__device__ __forceinline__ void decode_sub2(uint32_t w, uint32_t (&out)[8]) {
  const uint32_t w8 = w >> 8;
  out[0] = lop3_and_xor(w, 0x00030003u, 0x00020002u);
  out[1] = lop3_and_xor(w, 0x000C000Cu, 0x00080008u);
  out[2] = lop3_and_xor(w, 0x00300030u, 0x00200020u);
  out[3] = lop3_and_xor(w, 0x00C000C0u, 0x00800080u);
  out[4] = lop3_and_xor(w8, 0x00030003u, 0x00020002u);
  out[5] = lop3_and_xor(w8, 0x000C000Cu, 0x00080008u);
  out[6] = lop3_and_xor(w8, 0x00300030u, 0x00200020u);
  out[7] = lop3_and_xor(w8, 0x00C000C0u, 0x00800080u);
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// INT3 word -> one MMA register of fp16 subnormals: fields p and p + 5 (15
// bits apart) land at bits 1..3 and 16..18, i.e. (2 u_p, u_{p+5}) * 2^-24
// with u = code + 4 (the XOR flips each field's sign bit).  p is a constant
// after unrolling.
__device__ __forceinline__ uint32_t ext3(uint32_t w, int p) {
  const uint32_t sh = p == 0 ? (w << 1) : (w >> (3 * p - 1));
  return lop3_and_xor(sh, 0x0007000Eu, 0x00040008u);
}

__device__ __forceinline__ __half lds_f16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __ushort_as_half(v);
}

// Cost-balanced ranges of the flattened stage list.  A stage costs kUnit;
// the first stage of each segment (sequence, head group) costs kSegCost<W>
// more, for the segment's own fixed work (its Q rows, the cross-warp merge,
// the partial or output write), so a range that a segment boundary cuts gets
// fewer stages.  With C(gs) the summed cost of the stages before gs and
// Wc = C(T), CTA i of n owns the stages with t_i <= C(gs) < t_{i+1},
// t_i = floor(i * Wc / n); a range may be empty.
constexpr int64_t kUnit = 16;
template <int W>
constexpr int64_t kSegCost = W == 12 ? 14 : 12;

// Quotient of non-negative integers: 32-bit division when both fit (the
// common case, a few instructions), else 64-bit (a long software routine).
__host__ __device__ __forceinline__ int64_t udiv(int64_t a, int64_t b) {
  if (((a | b) >> 32) == 0) return static_cast<uint32_t>(a) / static_cast<uint32_t>(b);
  return a / b;
}
__host__ __device__ __forceinline__ int64_t cost_target(int64_t i, int64_t Wc, int64_t n) {
  return udiv(i * Wc, n);
}
// CTA owning the stage whose cost offset is x: the largest i with t_i <= x.
__host__ __device__ __forceinline__ int64_t cost_owner(int64_t x, int64_t Wc, int64_t n) {
  const int64_t i = udiv((x + 1) * n + Wc - 1, Wc) - 1;
  return i < n - 1 ? i : n - 1;
}
// Inside a segment the cost offset of stage g is 0 (g = 0), else sc + kUnit*g:
// the first stage g whose offset reaches rr.
__host__ __device__ __forceinline__ int64_t stage_at(int64_t rr, int64_t sc) {
  if (rr <= 0) return 0;
  if (rr <= sc + kUnit) return 1;
  return (rr - sc + kUnit - 1) / kUnit;  // kUnit = 16: a shift
}
// First stage of CTA i: prefix[b] = groups * (stages of sequences before b),
// nzp[b] = non-empty sequences before b, so the cost before sequence b is
// kUnit * prefix[b] + sc * groups * nzp[b].
__device__ __forceinline__ int64_t cost_start(int64_t i, int64_t n, int64_t Wc, const int *prefix, const int *nzp,
                                              int batch, int groups, int64_t sc) {
  const int64_t t = cost_target(i, Wc, n);
  if (t >= Wc) return prefix[batch];
  auto P = [&](int b) { return kUnit * prefix[b] + sc * groups * nzp[b]; };
  int lo = 0, hi = batch - 1;  // largest b with P(b) <= t: always a non-empty sequence
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P(mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int64_t nb = (prefix[lo + 1] - prefix[lo]) / groups;
  const int64_t L = sc + kUnit * nb;  // cost of one segment of sequence lo
  const int64_t r = t - P(lo), h = udiv(r, L);
  return prefix[lo] + h * nb + stage_at(r - h * L, sc);
}

struct Loc {
  int b, hg, s, n;  // sequence, head group, stage within the segment, stages of the segment
};

// prefix[b] = groups * (stages of sequences 0..b-1); locate the segment of gs.
__device__ __forceinline__ Loc locate(int64_t gs, const int *prefix, int batch, int groups) {
  int lo = 0, hi = batch - 1;  // largest b with prefix[b] <= gs: always a non-empty sequence
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= gs) lo = mid; else hi = mid - 1;
  }
  Loc l;
  l.b = lo;
  l.n = (prefix[lo + 1] - prefix[lo]) / groups;
  const int r = static_cast<int>(gs - prefix[lo]);
  l.hg = r / l.n;
  l.s = r - l.hg * l.n;
  return l;
}

// Fused append (TurboAttention §2.1: a decoding step appends k_t, v_t to the cache
// and attends over it).  The range holding the last stage of a segment
// quantizes that segment's new rows (k and v of each kv-head of the group)
// into the cache at position seq_lens[b] - 1, one consumer warp per row,
// while its producer streams the earlier stages; the producer loads the
// stage that holds them only after the consumers' `appended` barrier.  No
// other range reads those rows.  A new token beyond the cache (a clamped
// length) or in a missing page is not written.
template <int D>
__device__ void append_rows(const DecodeArgs &a, const KvView &cache, int hb, int groups, const int *prefix,
                            int64_t gs0, int64_t gs1, uint32_t *err, int warp, int lane, int nwarps) {
  const int64_t limit = cache.page_table ? static_cast<int64_t>(cache.max_pages) * kPage : cache.capacity;
  int item = 0;  // (segment, row) items of this range, dealt round-robin to the warps
  for (int64_t gs = gs0; gs < gs1;) {
    const Loc l = locate(gs, prefix, a.batch, groups);
    const int64_t last = gs - l.s + l.n - 1;  // the segment's last stage
    if (last < gs1) {
      const int64_t pos = static_cast<int64_t>(__ldg(a.seq_lens + l.b)) - 1;  // the new token
      for (int r = 0; r < 2 * hb; ++r, ++item) {
        if (item % nwarps != warp) continue;
        const int h = l.hg * hb + (r >> 1);
        int64_t dst = -1;
        if (pos >= limit) {
          // the length was clamped (and flagged) by the caller of this function
        } else if (!cache.page_table) {
          dst = (static_cast<int64_t>(l.b) * cache.hkv + h) * cache.capacity + pos;
        } else {
          const int page = __ldg(cache.page_table + static_cast<int64_t>(l.b) * cache.max_pages + pos / kPage);
          if (page >= 0 && page < cache.num_pages)
            dst = (static_cast<int64_t>(page) * cache.hkv + h) * kPage + pos % kPage;
          else if (lane == 0)
            atomicOr(err, kFlagBadPage);
        }
        if (dst < 0) continue;  // warp-uniform
        const bool is_v = r & 1;
        const int64_t src_row = static_cast<int64_t>(l.b) * cache.hkv + h;
        uint8_t *codes = (is_v ? cache.v_codes : cache.k_codes) + dst * (D / 2);
        uint16_t *scale = (is_v ? cache.v_scales : cache.k_scales) + dst;
        const void *src = is_v ? a.v_new : a.k_new;
        if (a.new_fp16)
          quantize_row_warp<__half, D>(static_cast<const __half *>(src) + src_row * D, codes, scale, lane);
        else
          quantize_row_warp<float, D>(static_cast<const float *>(src) + src_row * D, codes, scale, lane);
        // the rows are read back by this CTA's TMA loads (async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
    }
    gs = last + 1;
  }
}

// Geometry of one stage.  A TMA box streams at full speed only when its
// bytes are contiguous: in a contiguous cache a kv-head's tokens are, so a
// stage is 256 (W = 8) or 384 (W = 12) tokens of one kv-head; in a paged
// pool the kv-heads of a page are adjacent, so a stage is one page (64
// tokens) of 4 kv-heads (256/Hkv tokens of every head, page by page, when
// Hkv < 4; W = 8).
struct StageGeo {
  int hb;      // kv-heads per stage
  int tokens;  // tokens per head per stage = rows / hb
  int groups;  // head groups = Hkv / hb
  int wph;     // consumer warps per head = W / hb
};
template <int W>
__host__ __device__ __forceinline__ StageGeo stage_geo(int hkv, bool paged) {
  StageGeo g;
  g.hb = paged ? (hkv >= 4 ? 4 : hkv) : 1;
  g.tokens = Layout<W>::kRows / g.hb;
  g.groups = hkv / g.hb;
  g.wph = W / g.hb;
  return g;
}


// Tensor maps of one cache (built on the host, passed by value):
//   codes  3-D [heads_total][rows_per_head][128 B]; box [box_heads][box_rows][128 B], 128B swizzle
//   scales 2-D [heads_total][tokens_per_head] fp16; box [box_heads][box_tokens]
// heads_total = B*Hkv (contiguous) or P*Hkv (paged); a paged stage of more
// than one page is loaded page by page and head by head (box_heads = 1).
struct Maps {
  CUtensorMap k, v, ks, vs;
};

// ---------------------------------------------- segment cluster: merge CTAs
// Every thread of every CTA of the cluster reaches both cluster barriers once
// (the producer warps after their loads; `threads` consumer threads here).
// Between them, the segment's rows x D/4 float4 columns are shared out over
// the cluster; each reads the S partials (O rows, then the lse in log2 units,
// in the CTAs' Q slots) and writes out, lse.
template <int D>
__device__ __forceinline__ void cluster_merge(const DecodeArgs &a, const StageGeo &geo, int G, __half *qslot, bool empty,
                                           int threads) {
  const int S = a.cluster, rows = geo.hb * G;
  float *xo = reinterpret_cast<float *>(qslot);
  float *xl = xo + QATTN_MAX_GROUP * D;
  if (empty)  // no stage in this CTA: an empty partial
    for (int r = threadIdx.x; r < rows; r += threads) xl[r] = -INFINITY;
  cluster_sync();
  const uint32_t rank = cluster_rank();
  const int sg = blockIdx.x / S, b = sg / geo.groups, hg = sg - b * geo.groups;
  const uint32_t xo_a = smem_u32(xo), xl_a = smem_u32(xl);
  for (int it = static_cast<int>(rank) + S * threadIdx.x; it < rows * (D / 4); it += S * threads) {
    const int r = it / (D / 4), d = (it - r * (D / 4)) * 4;
    float lv[kMaxCluster];
    float M = -INFINITY;
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p) {
      lv[p] = p < S ? ld_dsmem_f32(dsmem_addr(xl_a + 4 * r, p)) : -INFINITY;
      M = fmaxf(M, lv[p]);
    }
    float Z = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p) {
      if (p < S && lv[p] != -INFINITY) {
        const float w = ex2(lv[p] - M);
        const float4 v = ld_dsmem_f32x4(dsmem_addr(xo_a + 4 * (r * D + d), p));
        Z += w;
        acc.x += w * v.x, acc.y += w * v.y, acc.z += w * v.z, acc.w += w * v.w;
      }
    }
    const bool live = Z > 0.f;
    const float inv = live ? 1.f / Z : 0.f;
    const int64_t row = static_cast<int64_t>(b) * a.hq + (hg * geo.hb + r / G) * G + r % G;
    const uint32_t h01 = pack_half2(acc.x * inv, acc.y * inv), h23 = pack_half2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(a.out + row * D + d) = make_uint2(h01, h23);
    if (d == 0 && a.lse) a.lse[row] = live ? (M + log2f(Z)) * 0.69314718055994531f : -INFINITY;
  }
  cluster_sync();  // the other CTAs have read this CTA's partial
}

template <int D, int W, int BITS = 4, bool kCluster = false>
__global__ void __launch_bounds__(Layout<W>::kThreads, 1)
    decode_kernel(DecodeArgs a, KvView cache, const __grid_constant__ Maps maps, uint32_t *err) {
  using C = Cfg<D, W, BITS>;
  constexpr int kConsumerWarps = W;
  constexpr int kThreads = Layout<W>::kThreads;
  constexpr int kRowsPerStage = Layout<W>::kRows;
  const int G = a.hq / cache.model_hkv;
  const int B = a.batch, hkv = cache.hkv;
  const StageGeo geo = stage_geo<W>(hkv, cache.page_table != nullptr);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __half *qslot = reinterpret_cast<__half *>(smem + C::kRing);      // [rows of a segment][D]
  float *smm = reinterpret_cast<float *>(smem + C::kRing + C::kQSlot);  // [warp][8]
  float *sml = smm + kConsumerWarps * 8;                              // [warp][8]
  int *prefix = reinterpret_cast<int *>(sml + kConsumerWarps * 8);    // [B + 1]
  int *lens = prefix + B + 1;                                         // [B], clamped
  int *nzp = lens + B;                                                // [B + 1], non-empty sequences before b
  uint64_t *full = reinterpret_cast<uint64_t *>(
      (reinterpret_cast<uintptr_t>(nzp + B + 1) + 7) & ~static_cast<uintptr_t>(7));
  uint64_t *empty = full + C::kStages;
  uint64_t *qfull = empty + C::kStages;
  uint64_t *qempty = qfull + 1;
  uint64_t *appended = qempty + 1;                                   // fused append done (consumer warps)
  int *valid = reinterpret_cast<int *>(appended + 1);                // [kStages]: 0 = missing page
  volatile int *abort_flag = valid + C::kStages;                     // set after a timed-out wait
  int64_t *range = reinterpret_cast<int64_t *>(valid + C::kStages + 2);  // [2]: this CTA's first, end stage

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool paged = cache.page_table != nullptr;
  const int64_t limit = paged ? static_cast<int64_t>(cache.max_pages) * kPage : cache.capacity;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kConsumerWarps);
    }
    mbar_init(smem_u32(qfull), 1);
    mbar_init(smem_u32(qempty), kConsumerWarps);
    mbar_init(smem_u32(appended), kConsumerWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == kConsumerWarps * 32) {  // descriptors are kernel parameters: fetch early
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
    prefetch_tmap(&maps.ks);
    prefetch_tmap(&maps.vs);
  }

  // Before the programmatic wait below, the kernels that may still be running
  // are this library's decode, merge and combine kernels of earlier calls on
  // the stream (the only ones that release their dependents early).  They
  // write cache rows (the fused append), partials, out and lse, never the
  // sequence lengths or the page table: so the lengths, the stage prefix and
  // this CTA's range are computed here, and its first stages are prefetched
  // into L2 (the point of coherence: a later write still wins).  Q and the
  // cache rows are read only after the wait.
  // prefix[b]: first global stage of sequence b (all its head groups)
  for (int b = threadIdx.x; b < B; b += kThreads) {
    int len = __ldg(a.seq_lens + b);
    if (len > limit) {
      len = static_cast<int>(limit);
      atomicOr(err, kFlagBadPage);
    }
    if (len < 0) len = 0;
    lens[b] = len;
    prefix[b + 1] = len > 0 ? geo.groups * ((len + geo.tokens - 1) / geo.tokens) : 0;
    nzp[b + 1] = len > 0;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0, carry_nz = 0;
    for (int base = 0; base < B; base += 32) {
      int v = base + lane < B ? prefix[base + lane + 1] : 0;
      int vn = base + lane < B ? nzp[base + lane + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        const int un = __shfl_up_sync(0xffffffffu, vn, o);
        if (lane >= o) v += u, vn += un;
      }
      if (base + lane < B) prefix[base + lane + 1] = carry + v, nzp[base + lane + 1] = carry_nz + vn;
      carry += __shfl_sync(0xffffffffu, v, 31);
      carry_nz += __shfl_sync(0xffffffffu, vn, 31);
    }
    if (lane == 0) prefix[0] = 0, nzp[0] = 0;
  }
  __syncthreads();

  const int64_t T = prefix[B];
  const int64_t sc = kSegCost<W>;
  const int64_t Wc = kUnit * T + sc * geo.groups * nzp[B];
  // The range is computed once per CTA, by two lanes of warp 0, and shared:
  // every thread computing it would keep the SM's issue slots busy with the
  // same divisions for longer than the extra barrier takes.
  // With segment clusters (a.cluster = S CTAs per (sequence, head group)
  // segment, CTAs k S .. k S + S - 1 forming cluster k), CTA rank r takes the
  // segment's stages [r n / S, (r + 1) n / S).
  if (warp == 0 && lane < 2) {
    if constexpr (kCluster) {
      const int S = a.cluster, sg = blockIdx.x / S, rk = blockIdx.x - sg * S + lane;
      const int b = sg / geo.groups, hg = sg - b * geo.groups;
      const int n = (prefix[b + 1] - prefix[b]) / geo.groups;
      range[lane] = prefix[b] + static_cast<int64_t>(hg) * n + static_cast<int64_t>(rk) * n / S;
    } else {
      range[lane] = cost_start(blockIdx.x + lane, gridDim.x, Wc, prefix, nzp, B, geo.groups, sc);
    }
  }
  __syncthreads();
  const int64_t gs0 = range[0], gs1 = range[1];
  if (!kCluster && gs1 <= gs0) return;  // (a cluster's CTAs all meet at its merge)
  // L2 prefetch of the range's first two stages while a preceding kernel may
  // still run (L2 is the coherence point: a later write still wins)
  if (!paged && threadIdx.x == kConsumerWarps * 32 + 1) {
    for (int k = 0; k < 2 && gs0 + k < gs1; ++k) {
      const Loc l = locate(gs0 + k, prefix, B, geo.groups);
      const int64_t tok0 = static_cast<int64_t>(l.s) * geo.tokens;
      const int64_t ntok = min(static_cast<int64_t>(geo.tokens), cache.capacity - tok0);
      const int64_t row = (static_cast<int64_t>(l.b) * hkv + l.hg * geo.hb) * cache.capacity + tok0;
      const uint32_t cb = static_cast<uint32_t>(ntok * C::kTokBytes), sb = static_cast<uint32_t>(ntok * 2);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(cache.k_codes + row * C::kTokBytes), "r"(cb) : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(cache.v_codes + row * C::kTokBytes), "r"(cb) : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(cache.k_scales + row), "r"(sb) : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(cache.v_scales + row), "r"(sb) : "memory");
    }
  }
  pdl_wait();                // cache rows and Q may come from the preceding kernel on the stream
  pdl_launch_dependents();   // the merge kernel may be scheduled as SMs free up

  if (warp >= kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // (layout W = 12: a warpgroup whose registers go to the consumers; one
    // thread of its first warp issues the loads)
    if constexpr (Layout<W>::kSplitRegs) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Layout<W>::kRegsProducer));
    // the loads; every way out of them (an abort included) reaches the
    // cluster barriers below
    if (warp == kConsumerWarps && lane == 0) {
      const int rows_per_tok = C::kTokBytes;  // code bytes per token
      const uint32_t qbytes = geo.hb * G * D * 2;
      int it = 0, seg = 0;
      bool rows_in = a.k_new == nullptr;  // the fused append's rows are in the cache
      for (int64_t gs = gs0; gs < gs1; ++seg) {
        const Loc l = locate(gs, prefix, B, geo.groups);
        const int cnt = static_cast<int>(min(static_cast<int64_t>(l.n - l.s), gs1 - gs));
        const int seg_len = lens[l.b];
        // the segment's Q rows (its head group's q-heads are contiguous)
        {
          if (seg >= 1 && !mbar_wait(smem_u32(qempty), (seg & 1) ^ 1, err,
                                     *abort_flag ? kDrainCycles : kWaitCycles)) {
            *abort_flag = 1;
            goto producer_done;
          }
          const uint32_t qf = smem_u32(qfull);
          int mh = model_head(cache.head_map, cache.model_hkv, l.hg * geo.hb);
          if (mh < 0) {  // no such model head: a harmless load; its rows are not written
            atomicOr(err, kFlagBadHead);
            mh = 0;
          }
          mbar_arrive_expect_tx(qf, qbytes);
          bulk_g2s(smem_u32(qslot), a.q + (static_cast<int64_t>(l.b) * a.hq + static_cast<int64_t>(mh) * G) * D, qbytes, qf);
        }
        for (int j = 0; j < cnt; ++j, ++it) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (it >= C::kStages &&
              !mbar_wait(smem_u32(empty + s), ph ^ 1, err, *abort_flag ? kDrainCycles : kWaitCycles)) {
            *abort_flag = 1;  // stop issuing; the consumers drain with short waits
            goto producer_done;
          }
          if (!rows_in && l.s + j == l.n - 1) {  // a segment's last stage holds its new rows
            rows_in = true;
            if (!mbar_wait(smem_u32(appended), 0, err, *abort_flag ? kDrainCycles : kWaitCycles)) {
              *abort_flag = 1;
              goto producer_done;
            }
          }
          const int tok0 = (l.s + j) * geo.tokens;  // first token of the stage in the sequence
          const uint32_t full_s = smem_u32(full + s);
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t stv = st + C::kCodeBytes, sks = st + 2 * C::kCodeBytes, svs = sks + C::kScaleBytes;
          const int head_base = l.hg * geo.hb;
          if (!paged) {
            const int head0 = l.b * hkv + head_base;
            const int row0 = tok0 * rows_per_tok / 128;
            valid[s] = 1;
            mbar_arrive_expect_tx(full_s, 2 * C::kCodeBytes + 2 * C::kScaleBytes);
            tma_load_3d(st, &maps.k, 0, row0, head0, full_s);
            tma_load_3d(stv, &maps.v, 0, row0, head0, full_s);
            // scale boxes are at most 256 tokens: a 384-token stage takes two
            constexpr int kSBox = kRowsPerStage > 256 ? kRowsPerStage / 2 : kRowsPerStage;
#pragma unroll
            for (int o = 0; o < kRowsPerStage; o += kSBox) {
              tma_load_2d(sks + 2 * o, &maps.ks, tok0 + o, head0, full_s);
              tma_load_2d(svs + 2 * o, &maps.vs, tok0 + o, head0, full_s);
            }
          } else {
            // pages of this stage that hold tokens below the sequence length
            // (a stage may run past the end of the sequence and of its table row)
            const int npages = geo.tokens > kPage ? geo.tokens / kPage : 1;
            const int nused = min(npages, (seg_len - tok0 + kPage - 1) / kPage);
            bool ok = true;
            for (int pi = 0; pi < nused; ++pi) {
              const int page = __ldg(cache.page_table + static_cast<int64_t>(l.b) * cache.max_pages +
                                     (tok0 + pi * kPage) / kPage);
              ok = ok && page >= 0 && page < cache.num_pages;
            }
            valid[s] = ok;
            if (!ok) {
              atomicOr(err, kFlagBadPage);
              mbar_arrive(full_s);  // a missing page: the stage's tokens are masked
              continue;
            }
            const uint32_t bytes = npages == 1
                ? 2 * C::kCodeBytes + 2 * C::kScaleBytes
                : nused * geo.hb * (2 * kPage * rows_per_tok + 2 * kPage * 2);
            mbar_arrive_expect_tx(full_s, bytes);
            for (int pi = 0; pi < nused; ++pi) {
              const int ptok = tok0 + pi * kPage;
              const int page = __ldg(cache.page_table + static_cast<int64_t>(l.b) * cache.max_pages + ptok / kPage);
              const int inner = ptok % kPage;  // token offset inside the page
              if (npages == 1) {               // every head of the stage in one box
                const int head0 = page * hkv + head_base;
                tma_load_3d(st, &maps.k, 0, inner * rows_per_tok / 128, head0, full_s);
                tma_load_3d(stv, &maps.v, 0, inner * rows_per_tok / 128, head0, full_s);
                tma_load_2d(sks, &maps.ks, inner, head0, full_s);
                tma_load_2d(svs, &maps.vs, inner, head0, full_s);
              } else {                         // one page of one head per box
                for (int h = 0; h < geo.hb; ++h) {
                  const int head = page * hkv + head_base + h;
                  const uint32_t cofs = (h * geo.tokens + pi * kPage) * rows_per_tok;
                  const uint32_t sofs = (h * geo.tokens + pi * kPage) * 2;
                  tma_load_3d(st + cofs, &maps.k, 0, 0, head, full_s);
                  tma_load_3d(stv + cofs, &maps.v, 0, 0, head, full_s);
                  tma_load_2d(sks + sofs, &maps.ks, 0, head, full_s);
                  tma_load_2d(svs + sofs, &maps.vs, 0, head, full_s);
                }
              }
            }
          }
        }
        gs += cnt;
      }
    }
  producer_done:
    if constexpr (kCluster) {  // the consumers' two cluster barriers, met by this warp too
      __syncwarp();
      cluster_sync();
      cluster_sync();
    }
    return;
  } else {  // each role sets its register budget inside its own branch

  // -------------------------------------------------------------- consumers
  if constexpr (Layout<W>::kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Layout<W>::kRegsConsumer));
  const int g = lane >> 2, c = lane & 3;
  const int hbw = warp / geo.wph;              // this warp's kv-head within the stage
  const int tok_w = (warp % geo.wph) * 32;     // its 32 tokens within that head's stage tokens
  const int kofs = hbw * geo.tokens * C::kTokBytes;  // byte offset of the head's codes in a stage
  const int sofs = hbw * geo.tokens;           // element offset of the head's scales
  const float kf = a.scale_log2 * kTwo24;      // folds the 2^-24 of the subnormal codes
  // Stage-relative swizzled offsets of this lane's K rows (tile t, rows g / g+8)
  // and of its ldmatrix.x4.trans rows (matrix q holds tokens (q & 2 ? 8 : 0) +
  // 0..7 of tile t at 16-byte chunk 2 jp + (q & 1)); the same in every stage.
  uint32_t koff[2][2], voff[2][D / 64];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      koff[t][h] = swz128(kofs + (tok_w + t * 16 + g + 8 * h) * C::kTokBytes + c * C::kKBytes);
#pragma unroll
    for (int jp = 0; jp < D / 64; ++jp) {
      const int q = lane >> 3;
      const int vt = tok_w + t * 16 + ((q & 2) ? 8 : 0) + (lane & 7);
      voff[t][jp] = swz128(kofs + vt * C::kTokBytes + (2 * jp + (q & 1)) * 16);  // INT2: jp = 0 only
    }
  }
  if (BITS == 4 && a.k_new) {
    // The fused append, while the producer fills the ring: the rows are
    // fenced to the async proxy, then released to the producer, which
    // loads no segment's last stage before this barrier completes.
    if constexpr (BITS == 4) append_rows<D>(a, cache, geo.hb, geo.groups, prefix, gs0, gs1, err, warp, lane, kConsumerWarps);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(appended));
  }
  const uint32_t ring = smem_u32(smem);
  int cur = 0;           // ring slot of the next stage
  uint32_t cur_ph = 0;   // its mbarrier parity
  int seg = 0;           // segment counter (Q slot parity)
  for (int64_t gs = gs0; gs < gs1; ++seg) {
    const Loc l = locate(gs, prefix, B, geo.groups);
    const int cnt = static_cast<int>(min(static_cast<int64_t>(l.n - l.s), gs1 - gs));
    const int len = lens[l.b];

    // Q of q-head g as the B operand, from the segment's Q rows in shared
    // memory.  Lane c covers d = c*D/4 + 8i + {0..7} (word i of its K code
    // bytes); the decoder pairs (e, e+4), and nibble positions 1 and 3 come
    // out 16x larger, so those columns carry q / 16.
    uint32_t qb[BITS == 3 ? C::kKs3 : C::kMt][2];
    float qsum = 0.f;
    if constexpr (BITS == 2) {
      // INT2: lane c covers d = 32 c + 16 i + {0..15} (word i of its K code
      // bytes); k-step 4 i + j multiplies fields (2j, 2j + 8) and (2j + 1,
      // 2j + 9) of the word, which come out 4^(e & 3) larger, so those
      // columns carry q / 4^(e & 3)
      if (!mbar_wait(smem_u32(qfull), seg & 1, err, *abort_flag ? kDrainCycles : kWaitCycles))
        *abort_flag = 1;
      const uint32_t qrow = smem_u32(qslot) + ((hbw * G + min(g, G - 1)) * D + c * (D / 4)) * 2;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 u = g < G ? lds128(qrow + 32 * i) : make_uint4(0, 0, 0, 0);
        const uint4 v = g < G ? lds128(qrow + 32 * i + 16) : make_uint4(0, 0, 0, 0);
        const uint32_t uu[4] = {u.x, u.y, u.z, u.w}, vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float s0 = (j & 1) ? 16.f : 1.f, s1 = (j & 1) ? 64.f : 4.f;
          const uint32_t e0 = __byte_perm(uu[j], vv[j], 0x5410), e1 = __byte_perm(uu[j], vv[j], 0x7632);
          const __half2 h0 = __hmul2(*reinterpret_cast<const __half2 *>(&e0), __float2half2_rn(1.f / s0));
          const __half2 h1 = __hmul2(*reinterpret_cast<const __half2 *>(&e1), __float2half2_rn(1.f / s1));
          qb[4 * i + j][0] = *reinterpret_cast<const uint32_t *>(&h0);
          qb[4 * i + j][1] = *reinterpret_cast<const uint32_t *>(&h1);
          const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
          qsum += s0 * (f0.x + f0.y) + s1 * (f1.x + f1.y);  // the values the MMA multiplies
        }
      }
    } else if constexpr (BITS == 3) {
      // INT3: register r of lane c takes field pair p = r % 5 of its word
      // slot r / 5 (words c, c + 4, c + 8, and 12 for lane 0): d = 10 w + p
      // (low half, which came out 2x larger: q / 2) and 10 w + p + 5
      if (!mbar_wait(smem_u32(qfull), seg & 1, err, *abort_flag ? kDrainCycles : kWaitCycles))
        *abort_flag = 1;
      const uint32_t qrow = smem_u32(qslot) + (hbw * G + min(g, G - 1)) * D * 2;
#pragma unroll
      for (int r = 0; r < 2 * C::kKs3; ++r) {
        const int jw = r / 5, p = r % 5;
        const int w = jw < 3 ? c + 4 * jw : (c == 0 ? 12 : -1);
        const int dlo = 10 * w + p, dhi = dlo + 5;
        float qlo = 0.f, qhi = 0.f;
        if (g < G && w >= 0) {
          if (dlo < D) qlo = __half2float(lds_f16(qrow + 2 * dlo));
          if (dhi < D) qhi = __half2float(lds_f16(qrow + 2 * dhi));
        }
        const __half2 h = __halves2half2(__float2half_rn(0.5f * qlo), __float2half_rn(qhi));
        qb[r >> 1][r & 1] = *reinterpret_cast<const uint32_t *>(&h);
        const float2 f = __half22float2(h);
        qsum += 2.f * f.x + f.y;  // the bias uses exactly the values the MMA multiplies
      }
    } else {
      if (!mbar_wait(smem_u32(qfull), seg & 1, err, *abort_flag ? kDrainCycles : kWaitCycles))
        *abort_flag = 1;
      const int dbase = c * (D / 4);
      const uint32_t qrow = smem_u32(qslot) + ((hbw * G + min(g, G - 1)) * D + dbase) * 2;
      const __half2 sixteenth = __float2half2_rn(0.0625f);
#pragma unroll
      for (int i = 0; i < C::kWords; ++i) {
        const uint4 u = g < G ? lds128(qrow + 16 * i) : make_uint4(0, 0, 0, 0);
        const uint32_t p0 = __byte_perm(u.x, u.z, 0x5410), p1 = __byte_perm(u.x, u.z, 0x7632);
        const uint32_t p2 = __byte_perm(u.y, u.w, 0x5410), p3 = __byte_perm(u.y, u.w, 0x7632);
        __half2 h1 = __hmul2(*reinterpret_cast<const __half2 *>(&p1), sixteenth);
        __half2 h3 = __hmul2(*reinterpret_cast<const __half2 *>(&p3), sixteenth);
        qb[2 * i][0] = p0;
        qb[2 * i][1] = *reinterpret_cast<uint32_t *>(&h1);
        qb[2 * i + 1][0] = p2;
        qb[2 * i + 1][1] = *reinterpret_cast<uint32_t *>(&h3);
        // the bias must use exactly the values the MMA multiplies
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&p0));
        const float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&p2));
        const float2 f1 = __half22float2(h1), f3 = __half22float2(h3);
        qsum += f0.x + f0.y + f2.x + f2.y + 16.f * (f1.x + f1.y + f3.x + f3.y);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(qempty));  // Q now lives in registers
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
    // raw-unit bias (code offset) * sum(q) * 2^-24 for the lane's q-heads 2c
    // and 2c+1; the offset is 8 for INT4 codes, 4 for INT3, 2 for INT2
    constexpr float kOff = BITS == 3 ? 4.f : BITS == 2 ? 2.f : 8.f;
    const float bq0 = kOff / kTwo24 * __shfl_sync(0xffffffffu, qsum, (2 * c) << 2);
    const float bq1 = kOff / kTwo24 * __shfl_sync(0xffffffffu, qsum, (2 * c + 1) << 2);

    float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f, ps0 = 0.f, ps1 = 0.f;
    float o[C::kOt][4];
#pragma unroll
    for (int mt = 0; mt < C::kOt; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    int last = 0;  // slot of the segment's last stage: its buffer hosts the merge
    for (int j = 0; j < cnt; ++j) {
      const bool got = mbar_wait(smem_u32(full + cur), cur_ph, err, *abort_flag ? kDrainCycles : kWaitCycles);
      if (!got) *abort_flag = 1;
      const int nvalid =
          (got && valid[cur]) ? max(0, min(len - (l.s + j) * geo.tokens - tok_w, 32)) : 0;
      if (nvalid > 0) {
        const uint32_t kb = ring + cur * C::kStageBytes;
        const uint32_t vb = kb + C::kCodeBytes;
        // scales by explicit shared-memory loads (the aligned base is not
        // known to the compiler as shared, generic loads would be slower)
        const uint32_t sks = kb + 2 * C::kCodeBytes + 2 * sofs;
        const uint32_t svs = sks + 2 * kRowsPerStage;
        // S^T of the warp's 32 tokens: two 16-token tiles, two accumulation
        // chains each (even / odd code words)
        float sacc[2][4], so[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[t][e] = so[t][e] = 0.f;
        if constexpr (BITS == 2) {
          // words 2c, 2c + 1 of rows g and g + 8 of each tile
          uint32_t kw[2][2][2];
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint2 u = lds64(kb + koff[t][h]);
              kw[t][h][0] = u.x, kw[t][h][1] = u.y;
            }
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              uint32_t x0[8], x1[8];
              decode_sub2(kw[t][0][i], x0);
              decode_sub2(kw[t][1][i], x1);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if (j & 1)
                  mma_16816(so[t], x0[2 * j], x1[2 * j], x0[2 * j + 1], x1[2 * j + 1], qb[4 * i + j][0], qb[4 * i + j][1]);
                else
                  mma_16816(sacc[t], x0[2 * j], x1[2 * j], x0[2 * j + 1], x1[2 * j + 1], qb[4 * i + j][0], qb[4 * i + j][1]);
              }
            }
        } else if constexpr (BITS == 3) {
          // words c, c + 4, c + 8 (and 12 for lane 0) of rows g and g + 8 of each tile
          uint32_t kw3[2][2][4];
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t rb = kb + kofs + (tok_w + 16 * t + g + 8 * h) * C::kTokBytes + 4 * c;
              kw3[t][h][0] = lds32(rb);
              kw3[t][h][1] = lds32(rb + 16);
              kw3[t][h][2] = lds32(rb + 32);
              kw3[t][h][3] = c == 0 ? lds32(rb + 48) : 0u;
            }
#pragma unroll
          for (int ks = 0; ks < C::kKs3; ++ks)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int r0 = 2 * ks, r1 = 2 * ks + 1;
              const uint32_t a0 = ext3(kw3[t][0][r0 / 5], r0 % 5), a1 = ext3(kw3[t][1][r0 / 5], r0 % 5);
              const uint32_t a2 = ext3(kw3[t][0][r1 / 5], r1 % 5), a3 = ext3(kw3[t][1][r1 / 5], r1 % 5);
              if (ks & 1)
                mma_16816(so[t], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
              else
                mma_16816(sacc[t], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            }
        } else {
        uint32_t kw[2][2][C::kWords];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if constexpr (C::kWords == 4) {
              const uint4 u = lds128(kb + koff[t][h]);
              kw[t][h][0] = u.x, kw[t][h][1] = u.y, kw[t][h][2] = u.z, kw[t][h][3] = u.w;
            } else {
              const uint2 u = lds64(kb + koff[t][h]);
              kw[t][h][0] = u.x, kw[t][h][1] = u.y;
            }
          }
#pragma unroll
        for (int i = 0; i < C::kWords; ++i)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            uint32_t x0[4], x1[4];
            decode_sub(kw[t][0][i], x0);
            decode_sub(kw[t][1][i], x1);
            if (i & 1) {
              mma_16816(so[t], x0[0], x1[0], x0[1], x1[1], qb[2 * i][0], qb[2 * i][1]);
              mma_16816(so[t], x0[2], x1[2], x0[3], x1[3], qb[2 * i + 1][0], qb[2 * i + 1][1]);
            } else {
              mma_16816(sacc[t], x0[0], x1[0], x0[1], x1[1], qb[2 * i][0], qb[2 * i][1]);
              mma_16816(sacc[t], x0[2], x1[2], x0[3], x1[3], qb[2 * i + 1][0], qb[2 * i + 1][1]);
            }
          }
        }
        float ts[2][4], fv[2][2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int lt = tok_w + t * 16 + g;
          const float f0 = __half2float(lds_f16(sks + 2 * lt)) * kf, f1 = __half2float(lds_f16(sks + 2 * lt + 16)) * kf;
          ts[t][0] = (sacc[t][0] + so[t][0] - bq0) * f0;
          ts[t][1] = (sacc[t][1] + so[t][1] - bq1) * f0;
          ts[t][2] = (sacc[t][2] + so[t][2] - bq0) * f1;
          ts[t][3] = (sacc[t][3] + so[t][3] - bq1) * f1;
          // the V scale carries an exact 2^-8: with a lazily raised max p can
          // reach 2^8, and p * s_V must stay inside the fp16 range
          fv[t][0] = __half2float(lds_f16(svs + 2 * lt)) * 0.00390625f;
          fv[t][1] = __half2float(lds_f16(svs + 2 * lt + 16)) * 0.00390625f;
        }
        if (nvalid < 32) {  // tail: mask tokens past the sequence end (never touch their scales)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const bool v0 = t * 16 + g < nvalid, v1 = t * 16 + g + 8 < nvalid;
            if (!v0) ts[t][0] = ts[t][1] = -INFINITY, fv[t][0] = 0.f;
            if (!v1) ts[t][2] = ts[t][3] = -INFINITY, fv[t][1] = 0.f;
          }
        }
        // lazy running max: rescale only when a score exceeds the max by 2^8
        const float lm0 = fmaxf(fmaxf(ts[0][0], ts[0][2]), fmaxf(ts[1][0], ts[1][2]));
        const float lm1 = fmaxf(fmaxf(ts[0][1], ts[0][3]), fmaxf(ts[1][1], ts[1][3]));
        if (__any_sync(0xffffffffu, lm0 > m0 + 8.f || lm1 > m1 + 8.f)) {
          float mx0 = lm0, mx1 = lm1;
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
          const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);
          m0 = n0, m1 = n1;
          l0 *= al0, l1 *= al1, ps0 *= al0, ps1 *= al1;
#pragma unroll
          for (int mt = 0; mt < C::kOt; ++mt) {
            o[mt][0] *= al0, o[mt][1] *= al1, o[mt][2] *= al0, o[mt][3] *= al1;
          }
        }
        uint32_t pb[2][2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float p0 = ex2(ts[t][0] - m0), p1 = ex2(ts[t][1] - m1);
          const float p2 = ex2(ts[t][2] - m0), p3 = ex2(ts[t][3] - m1);
          l0 += p0 + p2;
          l1 += p1 + p3;
          const uint32_t r0 = pack_half2(p0 * fv[t][0], p1 * fv[t][0]);
          const uint32_t r1 = pack_half2(p2 * fv[t][1], p3 * fv[t][1]);
          const float2 q0 = __half22float2(*reinterpret_cast<const __half2 *>(&r0));
          const float2 q1 = __half22float2(*reinterpret_cast<const __half2 *>(&r1));
          ps0 += q0.x + q1.x;  // sum of the fp16 P' the MMA sees (bias of the V codes)
          ps1 += q0.y + q1.y;
          pb[t][0] = movmatrix_trans(r0);
          pb[t][1] = movmatrix_trans(r1);
        }
        // O^T += V codes^T . P'^T
        if constexpr (BITS == 2) {
          // one ldmatrix.x4.trans per tile: matrix q holds tokens (q & 2 ? 8 :
          // 0) + 0..7 at 16-byte chunk q & 1 (64 dimensions); m-tile k row g
          // is d = 8 g + k, row g + 8 is d = 64 + 8 g + k (4^(k & 3) larger)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vb + voff[t][0], r0, r1, r2, r3);
            uint32_t d0[8], d1[8], d2[8], d3[8];
            decode_sub2(r0, d0);
            decode_sub2(r1, d1);
            decode_sub2(r2, d2);
            decode_sub2(r3, d3);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma_16816(o[k], d0[k], d1[k], d2[k], d3[k], pb[t][0], pb[t][1]);
          }
        } else if constexpr (BITS == 3) {
          // lane g owns words g and g + 8 of the V rows: m-tile 5 jj + p, row
          // g is d = 10 (g + 8 jj) + p (2x larger), row g + 8 is d + 5; the
          // two tokens of each A register come from two words, paired by
          // byte permutes of the two extractions
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            uint32_t vw[2][4];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int w = g + 8 * jj;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int tk = tok_w + 16 * t + 2 * c + (k & 1) + (k & 2 ? 8 : 0);
                vw[jj][k] = w < 13 ? lds32(vb + kofs + tk * C::kTokBytes + 4 * w) : 0u;
              }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
              for (int pp = 0; pp < 5; ++pp) {
                const uint32_t y0 = ext3(vw[jj][0], pp), y1 = ext3(vw[jj][1], pp);
                const uint32_t y2 = ext3(vw[jj][2], pp), y3 = ext3(vw[jj][3], pp);
                mma_16816(o[5 * jj + pp], __byte_perm(y0, y1, 0x5410), __byte_perm(y0, y1, 0x7632),
                          __byte_perm(y2, y3, 0x5410), __byte_perm(y2, y3, 0x7632), pb[t][0], pb[t][1]);
              }
          }
        } else {
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int jp = 0; jp < D / 64; ++jp) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vb + voff[t][jp], r0, r1, r2, r3);
            uint32_t d0[4], d1[4], d2[4], d3[4];
            decode_sub(r0, d0);
            decode_sub(r1, d1);
            decode_sub(r2, d2);
            decode_sub(r3, d3);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_16816(o[jp * 4 + k], d0[k], d1[k], d2[k], d3[k], pb[t][0], pb[t][1]);
          }
        }
      }
      __syncwarp();
      if (j + 1 < cnt) {
        if (lane == 0) mbar_arrive(smem_u32(empty + cur));
      } else {
        last = cur;  // released after the merge below
      }
      if (++cur == C::kStages) cur = 0, cur_ph ^= 1u;
    }

    // --------------------------------------------- segment end: merge warps
    // The last stage's buffer (every warp still holds it) becomes the merge
    // area: [warp][q-head][D + pad] fp32, written as float4 runs along d.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
    }
    consumer_sync<W>();  // every warp has read its last stage
    float *mo = reinterpret_cast<float *>(smem + last * C::kStageBytes);
    if constexpr (BITS == 2) {
      // O^T m-tile k: row g holds d = 8 g + k, row g + 8 holds d = 64 + 8 g + k,
      // 4^(k & 3) larger; code offset 2; P' carried 2^-8.  Float4 runs along d.
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int kg = 0; kg < 2; ++kg) {
          float v0[4], v1[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 4 * kg + e;
            const float f = kTwo24 / static_cast<float>(1 << (2 * (k & 3)));
            v0[e] = (o[k][2 * hh] * f - 2.f * ps0) * 256.f;
            v1[e] = (o[k][2 * hh + 1] * f - 2.f * ps1) * 256.f;
          }
          const int d = 64 * hh + 8 * g + 4 * kg;
          if (2 * c < G)
            *reinterpret_cast<float4 *>(mo + (warp * 8 + 2 * c) * C::kMergePitch + d) = make_float4(v0[0], v0[1], v0[2], v0[3]);
          if (2 * c + 1 < G)
            *reinterpret_cast<float4 *>(mo + (warp * 8 + 2 * c + 1) * C::kMergePitch + d) = make_float4(v1[0], v1[1], v1[2], v1[3]);
        }
    } else if constexpr (BITS == 3) {
      // O^T m-tile 5 jj + p: row g holds d = 10 (g + 8 jj) + p (2x larger),
      // row g + 8 holds d + 5; code offset 4; P' carried 2^-8
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int w = g + 8 * jj;
#pragma unroll
        for (int pp = 0; pp < 5; ++pp) {
          const int mt = 5 * jj + pp, dlo = 10 * w + pp, dhi = dlo + 5;
          if (w < 13 && dlo < D) {
            if (2 * c < G) mo[(warp * 8 + 2 * c) * C::kMergePitch + dlo] = (o[mt][0] * (kTwo24 / 2.f) - 4.f * ps0) * 256.f;
            if (2 * c + 1 < G)
              mo[(warp * 8 + 2 * c + 1) * C::kMergePitch + dlo] = (o[mt][1] * (kTwo24 / 2.f) - 4.f * ps1) * 256.f;
          }
          if (w < 13 && dhi < D) {
            if (2 * c < G) mo[(warp * 8 + 2 * c) * C::kMergePitch + dhi] = (o[mt][2] * kTwo24 - 4.f * ps0) * 256.f;
            if (2 * c + 1 < G) mo[(warp * 8 + 2 * c + 1) * C::kMergePitch + dhi] = (o[mt][3] * kTwo24 - 4.f * ps1) * 256.f;
          }
        }
      }
    } else {
    // O^T m-tile jp*4+k holds d = 64 jp + 4 g + k (rows g) and +32 (rows g+8);
    // nibble positions 1 and 3 (odd k) came out 16x larger; P' carried 2^-8.
#pragma unroll
    for (int jq = 0; jq < D / 32; ++jq) {  // d = 32 jq + 4 g + {0..3}
      const int jp = jq >> 1, hi = jq & 1;
      float4 v0, v1;
      v0.x = (o[jp * 4 + 0][2 * hi] * kTwo24 - 8.f * ps0) * 256.f;
      v0.y = (o[jp * 4 + 1][2 * hi] * (kTwo24 / 16.f) - 8.f * ps0) * 256.f;
      v0.z = (o[jp * 4 + 2][2 * hi] * kTwo24 - 8.f * ps0) * 256.f;
      v0.w = (o[jp * 4 + 3][2 * hi] * (kTwo24 / 16.f) - 8.f * ps0) * 256.f;
      v1.x = (o[jp * 4 + 0][2 * hi + 1] * kTwo24 - 8.f * ps1) * 256.f;
      v1.y = (o[jp * 4 + 1][2 * hi + 1] * (kTwo24 / 16.f) - 8.f * ps1) * 256.f;
      v1.z = (o[jp * 4 + 2][2 * hi + 1] * kTwo24 - 8.f * ps1) * 256.f;
      v1.w = (o[jp * 4 + 3][2 * hi + 1] * (kTwo24 / 16.f) - 8.f * ps1) * 256.f;
      const int d = 32 * jq + 4 * g;
      if (2 * c < G) *reinterpret_cast<float4 *>(mo + (warp * 8 + 2 * c) * C::kMergePitch + d) = v0;
      if (2 * c + 1 < G) *reinterpret_cast<float4 *>(mo + (warp * 8 + 2 * c + 1) * C::kMergePitch + d) = v1;
    }
    }
    if (g == 0) {
      smm[warp * 8 + 2 * c] = m0, smm[warp * 8 + 2 * c + 1] = m1;
      sml[warp * 8 + 2 * c] = l0, sml[warp * 8 + 2 * c + 1] = l1;
    }
    consumer_sync<W>();
    const bool complete = !kCluster && l.s == 0 && cnt == l.n;
    const int64_t pslot = l.s > 0 ? 2 * static_cast<int64_t>(blockIdx.x) : 2 * static_cast<int64_t>(blockIdx.x) + 1;
    // One thread per (row, 4 consecutive d): the row's warp weights
    // 2^(m_w - M) are computed once per thread, then 4 columns are folded
    // with float4 reads of the merge area.
    for (int idx = threadIdx.x; idx < geo.hb * G * (D / 4); idx += kConsumerWarps * 32) {
      const int r = idx / (D / 4), d = (idx - r * (D / 4)) * 4;  // row = kv-head in stage * G + q-head
      const int hh = r / G, h = r - hh * G;
      const int w0 = hh * geo.wph;
      // all warps' values are loaded before any is used (W is the bound of wph)
      float mw[W], lw[W];
      float4 xw[W];
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const bool in = w < geo.wph;
        const int k = (w0 + w) * 8 + h;
        mw[w] = in ? smm[k] : -INFINITY;
        lw[w] = in ? sml[k] : 0.f;
        xw[w] = in ? *reinterpret_cast<const float4 *>(mo + k * C::kMergePitch + d) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float M = mw[0];
#pragma unroll
      for (int w = 1; w < W; ++w) M = fmaxf(M, mw[w]);
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float sc = w < geo.wph ? ex2(mw[w] - M) : 0.f;
        L += sc * lw[w];
        acc.x += sc * xw[w].x, acc.y += sc * xw[w].y, acc.z += sc * xw[w].z, acc.w += sc * xw[w].w;
      }
      const bool live = L > 0.f;
      const float inv = live ? 1.f / L : 0.f;
      const float lse_v = live ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      if (complete) {
        const int mh = model_head(cache.head_map, cache.model_hkv, l.hg * geo.hb + hh);
        if (mh < 0) continue;  // flagged by the producer
        const int64_t row = static_cast<int64_t>(l.b) * a.hq + mh * G + h;
        const uint32_t h01 = pack_half2(acc.x * inv, acc.y * inv), h23 = pack_half2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(a.out + row * D + d) = make_uint2(h01, h23);
        if (d == 0 && a.lse) a.lse[row] = lse_v;
      } else if (kCluster) {
        // the cluster merge's input, in this CTA's Q slot (free once Q is in
        // registers; a cluster CTA has one segment): O rows, then the lse in
        // log2 units
        float *xo = reinterpret_cast<float *>(qslot);
        *reinterpret_cast<float4 *>(xo + r * D + d) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (d == 0) xo[QATTN_MAX_GROUP * D + r] = live ? M + log2f(L) : -INFINITY;
      } else {
        const int64_t prow = pslot * geo.hb * G + r;
        *reinterpret_cast<float4 *>(a.partial_o + prow * D + d) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (d == 0) a.partial_lse[prow] = lse_v;
      }
    }
    consumer_sync<W>();  // the merge area is read; the stage can be refilled
    if (lane == 0) mbar_arrive(smem_u32(empty + last));
    gs += cnt;
  }
  if constexpr (kCluster) cluster_merge<D>(a, geo, G, qslot, gs1 <= gs0, kConsumerWarps * 32);
  }
}

// Merges the partials of every (sequence, head-group) segment that the
// balanced ranges cut: a segment spanning CTAs c0 < c1 has partials in slot
// 2*c0 + 1 (its start, in c0's last segment) and slots 2*c for c0 < c <= c1
// whose range is not empty.  Segments of empty sequences get O = 0 and
// lse = -inf.  Two shapes, kWarps = 8 or 32:
//   8   grid (segments, rows of a segment): the 8 warps of a CTA split one
//       row's partials.  Small on purpose (256 threads, <= 64 registers, 4 KB
//       shared memory): beside an 8-warp decode CTA the programmatic launch
//       makes it resident while the decode still runs.  For few segments of
//       many partials (a long sequence cut into ~20 ranges per segment), the
//       rows spread over many SMs.
//   32  grid (segments): one 1024-thread CTA merges all rows of a segment,
//       32 / rows warps on each.  For many segments of 1-3 partials (a
//       batch of variable-length sequences), where launching and waiting for
//       one CTA per row costs more than the fold.
// A warp folds its partials with a running max so that the lse and O of a
// partial are fetched together, in batches of 4 whose loads are all issued
// before any is used; the warps of a row combine in shared memory.
template <int D, int W, int kWarps>
__global__ void __launch_bounds__(kWarps * 32, kWarps == 8 ? 4 : 1)
    decode_merge_kernel(const int32_t *__restrict__ seq_lens, int batch, int hkv, int G, int ctas,
                        int64_t limit, int paged, const int32_t *__restrict__ head_map, int model_hkv,
                        const float *__restrict__ po,
                        const float *__restrict__ pl, uint16_t *__restrict__ out,
                        float *__restrict__ lse) {
  constexpr int VPL = D / 32, KB = 4;
  __shared__ float accs[kWarps][D];
  __shared__ float wm[kWarps], wz[kWarps];
  __shared__ int redi[4][kWarps];
  const StageGeo geo = stage_geo<W>(hkv, paged != 0);
  const int b = blockIdx.x / geo.groups, hg = blockIdx.x % geo.groups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A programmatic dependent (the next decode on the stream) may be scheduled
  // now: before its own wait, which ends only once this grid has completed,
  // it reads only the sequence lengths and computes its range (nothing this
  // kernel writes) and prefetches into L2, so that work overlaps this merge.
  pdl_launch_dependents();
  // The decode kernel triggers this launch only after its own wait on the
  // inputs, so the lengths are final here; its partials are read after pdl_wait.
  auto stages = [&](int bb) {
    const int64_t len = min(static_cast<int64_t>(__ldg(seq_lens + bb)), limit);
    return len > 0 ? static_cast<int>((len + geo.tokens - 1) / geo.tokens) : 0;
  };
  // stages and non-empty sequences: in all, and before sequence b
  int tot = 0, pre = 0, nzt = 0, nzb = 0;
  for (int bb = threadIdx.x; bb < batch; bb += kWarps * 32) {
    const int n = stages(bb);
    tot += n, nzt += n > 0;
    if (bb < b) pre += n, nzb += n > 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    pre += __shfl_xor_sync(0xffffffffu, pre, o);
    nzt += __shfl_xor_sync(0xffffffffu, nzt, o);
    nzb += __shfl_xor_sync(0xffffffffu, nzb, o);
  }
  if (lane == 0) redi[0][warp] = tot, redi[1][warp] = pre, redi[2][warp] = nzt, redi[3][warp] = nzb;
  __syncthreads();
  tot = pre = nzt = nzb = 0;
  for (int w = 0; w < kWarps; ++w) tot += redi[0][w], pre += redi[1][w], nzt += redi[2][w], nzb += redi[3][w];
  const int rows = geo.hb * G;
  // this CTA's rows: one (kWarps = 8, grid.y = rows) or all of the segment's
  const int nr = kWarps == 8 ? 1 : rows, r0 = kWarps == 8 ? static_cast<int>(blockIdx.y) : 0;
  const int wpr = kWarps == 8 ? 8 : kWarps / rows;  // warps per row (rows <= 32)
  const int rl = warp / wpr, sub = warp - rl * wpr;
  auto out_row = [&](int r) {  // output row of segment row r; -1: no model head (flagged by the decode)
    const int mh = model_head(head_map, model_hkv, hg * geo.hb + r / G);
    return mh < 0 ? int64_t(-1) : (static_cast<int64_t>(b) * model_hkv + mh) * G + r % G;
  };
  const int n = stages(b);
  if (n == 0) {  // no decode CTA touches these rows
    pdl_wait();
    for (int i = threadIdx.x; i < nr * D; i += kWarps * 32) {
      const int64_t row = out_row(r0 + i / D);
      if (row < 0) continue;
      out[row * D + i % D] = 0;
      if (i % D == 0 && lse) lse[row] = -INFINITY;
    }
    return;
  }
  // the decode kernel's cost-balanced ranges: cost offsets of the segment's
  // first and last stages
  const int64_t sc = kSegCost<W>;
  const int64_t Wc = kUnit * geo.groups * tot + sc * geo.groups * nzt;
  const int64_t first = static_cast<int64_t>(geo.groups) * pre + static_cast<int64_t>(hg) * n;
  const int64_t cf = kUnit * geo.groups * pre + sc * geo.groups * nzb + hg * (sc + kUnit * n);
  const int64_t cl = n > 1 ? cf + sc + kUnit * (n - 1) : cf;
  const int64_t c0 = cost_owner(cf, Wc, ctas), c1 = cost_owner(cl, Wc, ctas);
  if (c0 == c1) return;  // finished inside one CTA
  const int np = static_cast<int>(c1 - c0 + 1);
  pdl_wait();
  float m = -INFINITY, z = 0.f, acc[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) acc[j] = 0.f;
  // Empty ranges (two 64-bit divisions to detect) exist only when a CTA's
  // share of the cost is below that of a segment's first stage; the starts
  // of CTAs c0 < c <= c1 + 1 are found from the segment's own cost offsets.
  const bool may_be_empty = Wc < (kUnit + sc) * ctas;
  auto start_in = [&](int64_t c) { return first + stage_at(cost_target(c, Wc, ctas) - cf, sc); };
  const int r = r0 + rl;
  if (rl < nr) {
    for (int k0 = sub; k0 < np; k0 += KB * wpr) {
      float lv[KB], x[KB][VPL];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int k = k0 + i * wpr;
        const int64_t c = c0 + k;
        const bool ok = k < np && (k == 0 || !may_be_empty || start_in(c) != start_in(c + 1));
        const int64_t slot = k == 0 ? 2 * c0 + 1 : 2 * c;
        lv[i] = ok ? pl[slot * rows + r] : -INFINITY;
        const float *src = po + (slot * rows + r) * D + lane * VPL;
        if constexpr (VPL == 4) {
          const float4 v = ok ? __ldg(reinterpret_cast<const float4 *>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
          x[i][0] = v.x, x[i][1] = v.y, x[i][2] = v.z, x[i][3] = v.w;
        } else {
          const float2 v = ok ? __ldg(reinterpret_cast<const float2 *>(src)) : make_float2(0.f, 0.f);
          x[i][0] = v.x, x[i][1] = v.y;
        }
      }
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        if (lv[i] == -INFINITY) continue;  // absent, or that split saw no key (its O is never used)
        const float mn = fmaxf(m, lv[i]);
        const float sc2 = expf(m - mn), e = expf(lv[i] - mn);
        z = z * sc2 + e;
#pragma unroll
        for (int j = 0; j < VPL; ++j) acc[j] = acc[j] * sc2 + e * x[i][j];
        m = mn;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j) accs[warp][lane * VPL + j] = acc[j];
  if (lane == 0) wm[warp] = m, wz[warp] = z;
  __syncthreads();
  for (int i = threadIdx.x; i < nr * D; i += kWarps * 32) {
    const int rr = i / D, d = i - rr * D, w0 = rr * wpr;
    float M = wm[w0];
    for (int w = 1; w < wpr; ++w) M = fmaxf(M, wm[w0 + w]);
    float Z = 0.f, o = 0.f;
    for (int w = 0; w < wpr; ++w) {
      if (wm[w0 + w] == -INFINITY) continue;
      const float e = expf(wm[w0 + w] - M);
      Z += wz[w0 + w] * e, o += accs[w0 + w][d] * e;
    }
    const int64_t row = out_row(r0 + rr);
    if (row < 0) continue;
    const float inv = M == -INFINITY ? 0.f : 1.f / Z;
    out[row * D + d] = __half_as_ushort(__float2half_rn(o * inv));
    if (d == 0 && lse) lse[row] = M == -INFINITY ? -INFINITY : M + logf(Z);
  }
}

cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  return attr;
}

// Segment clusters: with the split count left to the library, a contiguous
// cache without a head map, and at least two stages for each CTA, every
// (sequence, head group) segment gets a cluster of S = min(16, SMs /
// segments, stages) CTAs that merge through distributed shared memory: no
// merge kernel, no partials in global memory.  Taken only when every cluster
// of the grid can be resident at once (cudaOccupancyMaxActiveClusters, at the
// largest shared-memory size) and the grid covers at least 80 % of the SMs,
// else the cost-balanced ranges.
template <int D, int W, int BITS>
int cluster_size(bool auto_splits, bool paged, bool head_map, int batch, int hkv, int64_t max_len, int sms) {
  if (BITS != 4 || !auto_splits || paged || head_map) return 0;
  const StageGeo geo = stage_geo<W>(hkv, false);
  const int64_t segments = static_cast<int64_t>(batch) * geo.groups;
  const int64_t stages = (max_len + geo.tokens - 1) / geo.tokens;
  int64_t S = min(static_cast<int64_t>(kMaxCluster), min(sms / max(segments, int64_t(1)), stages));
  static int fits[kMaxCluster + 1] = {};  // per S: 0 unknown, else 1 + the resident clusters
  for (; S >= 2; --S) {
    if (fits[S] == 0) {
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = static_cast<unsigned>(S), at.val.clusterDim.y = 1, at.val.clusterDim.z = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(S));
      cfg.blockDim = dim3(Layout<W>::kThreads);
      cfg.dynamicSmemBytes = smem_bytes<D, W, BITS>(QATTN_MAX_BATCH);
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, W, BITS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           smem_bytes<D, W, BITS>(QATTN_MAX_BATCH));
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_kernel<D, W, BITS, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, decode_kernel<D, W, BITS, true>, &cfg);
      if (e != cudaSuccess) {
        cudaGetLastError();  // not an error of the call: the cost-balanced ranges are taken
        n = 0;
      }
      fits[S] = n + 1;
    }
    if (fits[S] - 1 >= segments)  // taken only if the clusters cover most of the SMs
      return 5 * segments * S >= 4 * static_cast<int64_t>(sms) ? static_cast<int>(S) : 0;
  }
  return 0;
}

template <int D, int W, int BITS = 4>
cudaError_t launch_d(const DecodeArgs &a0, const KvView &cache, const DecodeMaps &dm, uint32_t *err,
                     cudaStream_t stream) {
  static bool configured = false;  // per-function attributes, set once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, W, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes<D, W, BITS>(QATTN_MAX_BATCH));
    if constexpr (BITS == 4) {  // the segment-cluster form (INT4 only)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_kernel<D, W, BITS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes<D, W, BITS>(QATTN_MAX_BATCH));
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_kernel<D, W, BITS, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int G = a0.hq / cache.model_hkv;
  const bool paged = cache.page_table != nullptr;
  const StageGeo geo = stage_geo<W>(cache.hkv, paged);
  DecodeArgs a = a0;
  a.cluster = 0;
  if constexpr (BITS == 4)
    a.cluster = cluster_size<D, W, BITS>(a0.auto_splits != 0, paged, cache.head_map != nullptr, a0.batch, cache.hkv,
                                         min(static_cast<int64_t>(a0.max_len), cache.capacity), a0.sms);
  if (a.cluster > 0) a.ctas = a.batch * geo.groups * a.cluster;
  Maps maps;
  maps.k = dm.k, maps.v = dm.v, maps.ks = dm.ks, maps.vs = dm.vs;
  cudaLaunchAttribute attr[2] = {pdl_attr(), pdl_attr()};
  if (a.cluster > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(a.cluster), attr[1].val.clusterDim.y = 1, attr[1].val.clusterDim.z = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(Layout<W>::kThreads);
  cfg.dynamicSmemBytes = smem_bytes<D, W, BITS>(a.batch);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster > 0 ? 2 : 1;
  cudaError_t e;
  if constexpr (BITS == 4)
    e = a.cluster > 0 ? cudaLaunchKernelEx(&cfg, decode_kernel<D, W, BITS, true>, a, cache, maps, err)
                      : cudaLaunchKernelEx(&cfg, decode_kernel<D, W, BITS>, a, cache, maps, err);
  else
    e = cudaLaunchKernelEx(&cfg, decode_kernel<D, W, BITS>, a, cache, maps, err);
  if (e != cudaSuccess || a.cluster > 0) return e;
  const int64_t limit = cache.page_table ? static_cast<int64_t>(cache.max_pages) * kPage : cache.capacity;
  // one merge CTA per segment when segments are many (about two ranges or
  // fewer each), else one per row of a segment (rows = hb * G <= 32)
  const int64_t segments = static_cast<int64_t>(a.batch) * geo.groups;
  const bool per_segment = 2 * segments >= a.ctas;
  cudaLaunchConfig_t mc = {};
  mc.gridDim = dim3(static_cast<unsigned>(segments), per_segment ? 1 : geo.hb * G);
  mc.blockDim = dim3(per_segment ? 1024 : 256);
  mc.stream = stream;
  mc.attrs = attr;
  mc.numAttrs = 1;
  return cudaLaunchKernelEx(&mc, per_segment ? decode_merge_kernel<D, W, 32> : decode_merge_kernel<D, W, 8>,
                            a.seq_lens, a.batch, cache.hkv, G, a.ctas, limit,
                            static_cast<int>(paged), cache.head_map, static_cast<int>(cache.model_hkv),
                            static_cast<const float *>(a.partial_o), static_cast<const float *>(a.partial_lse),
                            a.out, a.lse);
}

}  // namespace

int decode_layout(int batch, int hkv, int max_len, bool paged, int ranges) {
  if (paged || ranges <= 0) return 8;
  const int64_t rows = static_cast<int64_t>(batch) * hkv * max_len;
  return rows >= static_cast<int64_t>(ranges) * 12 * Layout<12>::kRows ? 12 : 8;
}

DecodeGeometry decode_geometry(int head_dim, int hkv, bool paged, int warps) {
  const StageGeo g = (paged || warps == 8) ? stage_geo<8>(hkv, paged) : stage_geo<12>(hkv, false);
  DecodeGeometry r;
  r.heads_per_stage = g.hb;
  r.tokens_per_stage = g.tokens;
  r.groups = g.groups;
  const bool split_pages = paged && g.tokens > kPage;
  r.box_heads = split_pages ? 1 : g.hb;
  // TMA boxes hold at most 256 elements per dimension: a 384-token contiguous
  // stage loads its scales as two boxes of 192 (its codes, 192 rows of 128 B,
  // stay one box)
  r.box_tokens = paged ? (g.tokens > kPage ? kPage : g.tokens) : (g.tokens > 256 ? g.tokens / 2 : g.tokens);
  r.box_rows = (paged ? r.box_tokens : g.tokens) * head_dim / 256;
  return r;
}

int decode_cluster(int head_dim, int warps, int bits, bool auto_splits, bool paged, bool head_map, int batch,
                   int hkv, int64_t max_len, int sms) {
  if (bits != 4) return 0;
  if (head_dim == 128)
    return warps == 8 ? cluster_size<128, 8, 4>(auto_splits, paged, head_map, batch, hkv, max_len, sms)
                      : cluster_size<128, 12, 4>(auto_splits, paged, head_map, batch, hkv, max_len, sms);
  return warps == 8 ? cluster_size<64, 8, 4>(auto_splits, paged, head_map, batch, hkv, max_len, sms)
                    : cluster_size<64, 12, 4>(auto_splits, paged, head_map, batch, hkv, max_len, sms);
}

cudaError_t launch_decode(const DecodeArgs &a, const KvView &cache, const DecodeMaps &maps, uint32_t *err,
                          cudaStream_t stream) {
  if (a.batch == 0 || a.ctas <= 0) return cudaSuccess;
  if (cache.bits == 3)  // contiguous, D = 128
    return a.warps == 8 ? launch_d<128, 8, 3>(a, cache, maps, err, stream) : launch_d<128, 12, 3>(a, cache, maps, err, stream);
  if (cache.bits == 2)
    return a.warps == 8 ? launch_d<128, 8, 2>(a, cache, maps, err, stream) : launch_d<128, 12, 2>(a, cache, maps, err, stream);
  if (cache.page_table || a.warps == 8)
    return cache.head_dim == 128 ? launch_d<128, 8>(a, cache, maps, err, stream)
                                 : launch_d<64, 8>(a, cache, maps, err, stream);
  return cache.head_dim == 128 ? launch_d<128, 12>(a, cache, maps, err, stream)
                               : launch_d<64, 12>(a, cache, maps, err, stream);
}

}  // namespace qattn
