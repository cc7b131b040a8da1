// decode.cu -- split-KV decode attention over the INT4 cache.
//
// TurboAttention (arXiv 2412.08585) §2.1: a decode step attends the new query
// q_t against the whole cache; §2.2: FlashAttention's tiling with the online
// softmax of Milakov & Gimelshein (running max and sum, rescaling, final
// normalisation).  "Quantized Cross-Attention ... In-SRAM Dequantization"
// §3.1-§3.2: the 4-bit tile is brought from HBM into shared memory and
// dequantized inline, never written back as fp16; a quantized tile is 4x
// smaller, so a deeper ring of tiles fits on chip.
//
// Grid (splits, Hkv, B); a CTA owns the keys [split*chunk, (split+1)*chunk)
// of one (sequence, kv-head) and all G = Hq/Hkv query heads that read it.
//   warp 4       producer: per 64-token stage, two 2-D TMA loads of the K/V
//                codes (128-byte rows, 128B swizzle) and two bulk copies of
//                the K/V scales, completion tracked by an mbarrier ring.
//   warps 0-3    consumers: 16 tokens each per stage.
//     S^T (16 tokens x 8 heads) = codes_K (16 x D) . Q^T on mma.sync
//       m16n8k16 with tokens on M, the nibbles decoded to exact fp16
//       integers in registers; the fp32 result is multiplied by the
//       per-token K scale (exact scale folding, no fp16 rounding of c*s).
//     online softmax in the log2 domain, warp-uniform lazy rescale.
//     P' = P * s_V (per-token V scale folded into the probabilities), moved
//       to the B-operand layout with movmatrix.
//     O^T (D x 8 heads) += codes_V^T (D x 16 tokens) . P'^T, the V codes
//       transposed by ldmatrix.trans (pairs of tokens per register) and
//       decoded in registers.
//   end: the four consumer warps merge their (m, l, O) in shared memory; the
//   CTA writes the final fp16 O and lse (one split) or fp32 partials.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace qattn {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;

template <int D>
struct Cfg {
  static constexpr int kCodeBytes = kPage * D / 2;                          // per tensor
  static constexpr int kStageBytes = (2 * kCodeBytes + 4 * kPage + 1023) / 1024 * 1024;
  static constexpr int kKBytes = D / 8;  // K code bytes per lane per token
  static constexpr int kWords = kKBytes / 4;
  static constexpr int kMt = D / 16;     // m-tiles of O^T (and k-steps of S)
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 128;
  static_assert(kConsumerWarps * (8 * D + 16) * 4 <= kStages * kStageBytes, "merge scratch");
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(DecodeArgs a, KvView cache, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, uint32_t *err) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * C::kStageBytes);
  uint64_t *empty = full + kStages;
  int *valid = reinterpret_cast<int *>(empty + kStages);

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = a.hq / cache.hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool paged = cache.page_table != nullptr;

  int len = __ldg(a.seq_lens + b);
  const int64_t limit = paged ? static_cast<int64_t>(cache.max_pages) * kPage : cache.capacity;
  if (len > limit) {
    len = static_cast<int>(limit);
    if (threadIdx.x == 0 && split == 0 && kvh == 0) atomicOr(err, kFlagBadPage);
  }
  if (len < 0) len = 0;
  const int t_begin = split * a.chunk;
  const int t_end = min(t_begin + a.chunk, len);
  const int nst = t_end > t_begin ? (t_end - t_begin + kPage - 1) / kPage : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nst > 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      for (int it = 0; it < nst; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (it >= kStages && !mbar_wait(smem_u32(empty + s), ph ^ 1, err)) break;
        const int tok = t_begin + it * kPage;
        int64_t row_tok;  // cache row of the stage's first token
        bool ok = true;
        if (paged) {
          const int page = __ldg(cache.page_table + static_cast<int64_t>(b) * cache.max_pages + tok / kPage);
          ok = page >= 0 && page < cache.num_pages;
          if (!ok) atomicOr(err, kFlagBadPage);
          row_tok = (static_cast<int64_t>(ok ? page : 0) * cache.hkv + kvh) * kPage;
        } else {
          row_tok = (static_cast<int64_t>(b) * cache.hkv + kvh) * cache.capacity + tok;
        }
        valid[s] = ok;
        const uint32_t full_s = smem_u32(full + s);
        if (ok) {
          uint8_t *st = smem + s * C::kStageBytes;
          const int row128 = static_cast<int>(row_tok * (D / 2) / 128);
          mbar_arrive_expect_tx(full_s, 2 * C::kCodeBytes + 4 * kPage);
          tma_load_2d(smem_u32(st), &kmap, 0, row128, full_s);
          tma_load_2d(smem_u32(st + C::kCodeBytes), &vmap, 0, row128, full_s);
          bulk_g2s(smem_u32(st + 2 * C::kCodeBytes), cache.k_scales + row_tok, 2 * kPage, full_s);
          bulk_g2s(smem_u32(st + 2 * C::kCodeBytes + 2 * kPage), cache.v_scales + row_tok,
                   2 * kPage, full_s);
        } else {
          mbar_arrive(full_s);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  // Q as the B operand (k = head dim, n = head g).  The head-dim order inside
  // a k-step follows the nibble decoder: word i of lane c's code bytes covers
  // d = dbase + 8i + {0..7} and decode_nibbles yields the pairs (e, e + 4).
  uint32_t qb[C::kMt][2];
  {
    const int dbase = c * (D / 4);
    const __half *qrow =
        reinterpret_cast<const __half *>(a.q) + (static_cast<int64_t>(b) * a.hq + kvh * G + g) * D;
#pragma unroll
    for (int i = 0; i < C::kWords; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __half lo = __float2half(0.f), hi = __float2half(0.f);
        if (g < G) {
          lo = qrow[dbase + 8 * i + e];
          hi = qrow[dbase + 8 * i + e + 4];
        }
        __half2 h2 = __halves2half2(lo, hi);
        qb[2 * i + (e >> 1)][e & 1] = *reinterpret_cast<uint32_t *>(&h2);
      }
  }

  float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f;  // heads 2c, 2c+1 (log2 domain)
  float o[C::kMt][4];
#pragma unroll
  for (int mt = 0; mt < C::kMt; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int it = 0; it < nst; ++it) {
    const int s = it % kStages;
    const uint32_t ph = (it / kStages) & 1;
    if (!mbar_wait(smem_u32(full + s), ph, err)) break;
    const int nvalid = t_end - (t_begin + it * kPage + warp * 16);
    if (valid[s] && nvalid > 0) {
      const uint32_t kb = smem_u32(smem + s * C::kStageBytes);
      const uint32_t vb = kb + C::kCodeBytes;
      const __half *sks = reinterpret_cast<const __half *>(smem + s * C::kStageBytes + 2 * C::kCodeBytes);
      const __half *svs = sks + kPage;
      const int lt = warp * 16 + g;  // stage-local token of fragment row g

      // S^T = codes_K . Q^T  (rows g and g+8 = tokens lt, lt+8)
      uint32_t kw0[C::kWords], kw1[C::kWords];
      if constexpr (C::kWords == 4) {
        uint4 u0 = lds128(kb + swz128(lt * (D / 2) + c * C::kKBytes));
        uint4 u1 = lds128(kb + swz128((lt + 8) * (D / 2) + c * C::kKBytes));
        kw0[0] = u0.x, kw0[1] = u0.y, kw0[2] = u0.z, kw0[3] = u0.w;
        kw1[0] = u1.x, kw1[1] = u1.y, kw1[2] = u1.z, kw1[3] = u1.w;
      } else {
        uint2 u0 = lds64(kb + swz128(lt * (D / 2) + c * C::kKBytes));
        uint2 u1 = lds64(kb + swz128((lt + 8) * (D / 2) + c * C::kKBytes));
        kw0[0] = u0.x, kw0[1] = u0.y;
        kw1[0] = u1.x, kw1[1] = u1.y;
      }
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < C::kWords; ++i) {
        uint32_t x0[4], x1[4];
        decode_nibbles(kw0[i], x0);
        decode_nibbles(kw1[i], x1);
        mma_16816(sacc, x0[0], x1[0], x0[1], x1[1], qb[2 * i][0], qb[2 * i][1]);
        mma_16816(sacc, x0[2], x1[2], x0[3], x1[3], qb[2 * i + 1][0], qb[2 * i + 1][1]);
      }
      const bool v0 = g < nvalid, v1 = g + 8 < nvalid;
      const float fk0 = __half2float(sks[lt]) * a.scale_log2;
      const float fk1 = __half2float(sks[lt + 8]) * a.scale_log2;
      const float t0 = v0 ? sacc[0] * fk0 : -INFINITY, t1 = v0 ? sacc[1] * fk0 : -INFINITY;
      const float t2 = v1 ? sacc[2] * fk1 : -INFINITY, t3 = v1 ? sacc[3] * fk1 : -INFINITY;

      // online softmax: the running max changes rarely, so the rescale is a
      // warp-uniform branch taken only when some head's max grows.
      float mx0 = fmaxf(t0, t2), mx1 = fmaxf(t1, t3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      if (__any_sync(0xffffffffu, mx0 > m0 || mx1 > m1)) {
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);
        m0 = n0, m1 = n1, l0 *= al0, l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < C::kMt; ++mt) {
          o[mt][0] *= al0, o[mt][1] *= al1, o[mt][2] *= al0, o[mt][3] *= al1;
        }
      }
      const float p0 = ex2(t0 - m0), p1 = ex2(t1 - m1), p2 = ex2(t2 - m0), p3 = ex2(t3 - m1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      const float fv0 = v0 ? __half2float(svs[lt]) : 0.f;
      const float fv1 = v1 ? __half2float(svs[lt + 8]) : 0.f;
      const uint32_t pb0 = movmatrix_trans(pack_half2(p0 * fv0, p1 * fv0));
      const uint32_t pb1 = movmatrix_trans(pack_half2(p2 * fv1, p3 * fv1));

      // O^T += codes_V^T . P'^T: matrix q of ldmatrix.x4.trans holds tokens
      // (q & 2 ? 8 : 0) + 0..7 of this warp's slice at 16-byte chunk 2 jp + (q & 1).
#pragma unroll
      for (int jp = 0; jp < D / 64; ++jp) {
        const int q = lane >> 3;
        const int vt = warp * 16 + ((q & 2) ? 8 : 0) + (lane & 7);
        uint32_t r0, r1, r2, r3;
        ldsm_x4_trans(vb + swz128(vt * (D / 2) + (2 * jp + (q & 1)) * 16), r0, r1, r2, r3);
        uint32_t d0[4], d1[4], d2[4], d3[4];
        decode_nibbles(r0, d0);
        decode_nibbles(r1, d1);
        decode_nibbles(r2, d2);
        decode_nibbles(r3, d3);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_16816(o[jp * 4 + k], d0[k], d1[k], d2[k], d3[k], pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }

#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }

  // ------------------------------------------- merge the consumer warps
  consumer_sync();  // every warp is done with the stage buffers
  float *smo = reinterpret_cast<float *>(smem);  // [warp][head 8][D]
  float *smm = smo + kConsumerWarps * 8 * D;    // [warp][head 8]
  float *sml = smm + kConsumerWarps * 8;
#pragma unroll
  for (int jp = 0; jp < D / 64; ++jp)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int mt = jp * 4 + k;
      const int dlo = 64 * jp + 4 * g + k, dhi = dlo + 32;
      float *w0 = smo + (warp * 8 + 2 * c) * D;
      w0[dlo] = o[mt][0];
      w0[D + dlo] = o[mt][1];
      w0[dhi] = o[mt][2];
      w0[D + dhi] = o[mt][3];
    }
  if (g == 0) {
    smm[warp * 8 + 2 * c] = m0, smm[warp * 8 + 2 * c + 1] = m1;
    sml[warp * 8 + 2 * c] = l0, sml[warp * 8 + 2 * c + 1] = l1;
  }
  consumer_sync();
  const int tid = threadIdx.x;
  for (int idx = tid; idx < G * D; idx += kConsumerWarps * 32) {
    const int h = idx / D, d = idx % D;
    float M = smm[h];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) M = fmaxf(M, smm[w * 8 + h]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float sc = ex2(smm[w * 8 + h] - M);
      L += sc * sml[w * 8 + h];
      acc += sc * smo[(w * 8 + h) * D + d];
    }
    const int64_t row = static_cast<int64_t>(b) * a.hq + kvh * G + h;
    const bool live = L > 0.f;
    const float lse_v = live ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    if (a.splits == 1) {
      a.out[row * D + d] = __half_as_ushort(__float2half_rn(live ? acc / L : 0.f));
      if (d == 0 && a.lse) a.lse[row] = lse_v;
    } else {
      const int64_t prow = static_cast<int64_t>(split) * a.batch * a.hq + row;
      a.partial_o[prow * D + d] = live ? acc / L : 0.f;
      if (d == 0) a.partial_lse[prow] = lse_v;
    }
  }
}

template <int D>
cudaError_t launch_d(const DecodeArgs &a, const KvView &cache, const CUtensorMap &kmap,
                     const CUtensorMap &vmap, uint32_t *err, cudaStream_t stream) {
  using C = Cfg<D>;
  static bool configured = false;  // attribute is per-function, set once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(a.splits, cache.hkv, a.batch);
  decode_kernel<D><<<grid, kThreads, C::kSmem, stream>>>(a, cache, kmap, vmap, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, const KvView &cache, const CUtensorMap &kmap,
                          const CUtensorMap &vmap, uint32_t *err, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  return cache.head_dim == 128 ? launch_d<128>(a, cache, kmap, vmap, err, stream)
                               : launch_d<64>(a, cache, kmap, vmap, err, stream);
}

}  // namespace qattn
