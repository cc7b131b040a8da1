// prefill.cu -- causal prefill attention over the INT4 cache (warp-MMA path).
//
// TurboAttention (arXiv 2412.08585) §2.1 (prefill over the cached K, V) and
// §2.2 (FlashAttention: Q, K, V chunked along tokens, partial attention per
// pair of chunks, online max and sum, final normalisation).  The K/V tiles
// arrive as 4-bit codes plus per-token scales and are dequantized in
// registers right before the MMA ("Quantized Cross-Attention ... In-SRAM
// Dequantization" §3.1); no fp16 K/V is ever written to HBM.
//
// Grid (ceil(Nq/128), Hq, B), heaviest causal row blocks first.  A CTA owns
// 128 query rows of one head: eight consumer warps of 16 rows, and one
// producer warp streaming 64-token K/V stages (TMA, 128B swizzle) through an
// mbarrier ring shared with the decode kernel's layout.
//   S (16 x 8 tokens) = Q (16 x D) . codes_K^T : mma.sync m16n8k16, the K
//     nibbles of one token decoded into the B operand (pairs along D).
//   s = S * s_K[token] * scale * log2(e); causal / bounds mask; online softmax.
//   O (16 x D) += (P * s_V[token]) . codes_V : the probabilities reuse the S
//     accumulators as the A operand; V codes transposed by ldmatrix.trans.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace qattn {
namespace {

constexpr int kWarps = 8;                   // consumer warps (16 rows each)
constexpr int kRows = kWarps * 16;          // query rows per CTA
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kStages = 4;

template <int D>
struct PCfg {
  static constexpr int kCodeBytes = kPage * D / 2;
  static constexpr int kStageBytes = (2 * kCodeBytes + 4 * kPage + 1023) / 1024 * 1024;
  static constexpr int kQStride = D + 8;    // halves; padded rows of the staged Q tile
  static constexpr int kQBytes = kRows * kQStride * 2;
  static constexpr int kSmem = kStages * kStageBytes + kQBytes + 1024 + 128;
  static constexpr int kKs = D / 16;        // k-steps of S
  static constexpr int kWords = D / 32;     // K code words per lane per token
  static constexpr int kNt = D / 8;         // n-tiles of O
};

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(PrefillArgs a, KvView cache, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, uint32_t *err) {
  using C = PCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __half *sq = reinterpret_cast<__half *>(smem + kStages * C::kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * C::kStageBytes + C::kQBytes);
  uint64_t *empty = full + kStages;

  const int qblk = gridDim.x - 1 - blockIdx.x;  // longest causal blocks launch first
  const int hq = blockIdx.y, b = blockIdx.z;
  const int G = a.hq / cache.hkv, kvh = hq / G;
  const int q0 = qblk * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int shift = a.nk - a.nq;  // bottom-right causal alignment
  // keys this block can see: [0, kv_end)
  const int kv_end = a.causal ? min(a.nk, q0 + kRows + shift) : a.nk;
  const int ntiles = kv_end > 0 ? (kv_end + kPage - 1) / kPage : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && ntiles > 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      const int64_t base_tok = (static_cast<int64_t>(b) * cache.hkv + kvh) * cache.capacity;
      for (int it = 0; it < ntiles; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (it >= kStages && !mbar_wait(smem_u32(empty + s), ph ^ 1, err)) break;
        const int64_t row_tok = base_tok + static_cast<int64_t>(it) * kPage;
        const int row128 = static_cast<int>(row_tok * (D / 2) / 128);
        uint8_t *st = smem + s * C::kStageBytes;
        const uint32_t full_s = smem_u32(full + s);
        mbar_arrive_expect_tx(full_s, 2 * C::kCodeBytes + 4 * kPage);
        tma_load_2d(smem_u32(st), &kmap, 0, row128, full_s);
        tma_load_2d(smem_u32(st + C::kCodeBytes), &vmap, 0, row128, full_s);
        bulk_g2s(smem_u32(st + 2 * C::kCodeBytes), cache.k_scales + row_tok, 2 * kPage, full_s);
        bulk_g2s(smem_u32(st + 2 * C::kCodeBytes + 2 * kPage), cache.v_scales + row_tok, 2 * kPage,
                 full_s);
      }
    }
    return;
  }

  // ------------------------------------------------- stage Q through smem
  const __half *qg = reinterpret_cast<const __half *>(a.q) +
                     ((static_cast<int64_t>(b) * a.hq + hq) * a.nq) * D;
  for (int idx = threadIdx.x; idx < kRows * D / 8; idx += kWarps * 32) {
    const int r = idx / (D / 8), c8 = idx % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (q0 + r < a.nq) v = __ldg(reinterpret_cast<const uint4 *>(qg + static_cast<int64_t>(q0 + r) * D) + c8);
    *reinterpret_cast<uint4 *>(sq + r * C::kQStride + c8 * 8) = v;
  }
  consumers_sync();

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2, c = lane & 3;
  const int lr = warp * 16 + g;  // local rows lr, lr + 8
  // Q as the A operand.  Inside a k-step the head-dim order follows the K
  // nibble decoder: lane c's K code word i covers d = dbase + 8i + {0..7},
  // and decode_nibbles pairs (e, e + 4) for e = 0..3.
  uint32_t qa[C::kKs][4];
  {
    const int dbase = c * (D / 4);
#pragma unroll
    for (int i = 0; i < C::kWords; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d0 = dbase + 8 * i + e, ks = 2 * i + (e >> 1), slot = e & 1;
        __half2 h0 = __halves2half2(sq[lr * C::kQStride + d0], sq[lr * C::kQStride + d0 + 4]);
        __half2 h1 = __halves2half2(sq[(lr + 8) * C::kQStride + d0], sq[(lr + 8) * C::kQStride + d0 + 4]);
        qa[ks][2 * slot] = *reinterpret_cast<uint32_t *>(&h0);
        qa[ks][2 * slot + 1] = *reinterpret_cast<uint32_t *>(&h1);
      }
  }
  const int row0 = q0 + lr, row1 = row0 + 8;  // global query rows
  float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f;
  float o[C::kNt][4];
#pragma unroll
  for (int n = 0; n < C::kNt; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  for (int it = 0; it < ntiles; ++it) {
    const int s = it % kStages;
    const uint32_t ph = (it / kStages) & 1;
    if (!mbar_wait(smem_u32(full + s), ph, err)) break;
    const int tok0 = it * kPage;
    const bool any = !a.causal || tok0 <= q0 + warp * 16 + 15 + shift;
    if (any) {
      const uint32_t kb = smem_u32(smem + s * C::kStageBytes);
      const uint32_t vb = kb + C::kCodeBytes;
      const __half *sks = reinterpret_cast<const __half *>(smem + s * C::kStageBytes + 2 * C::kCodeBytes);
      const __half *svs = sks + kPage;
      float t[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t addr = kb + swz128((nt * 8 + g) * (D / 2) + c * (D / 8));
        uint32_t kw[C::kWords];
        if constexpr (C::kWords == 4) {
          uint4 u = lds128(addr);
          kw[0] = u.x, kw[1] = u.y, kw[2] = u.z, kw[3] = u.w;
        } else {
          uint2 u = lds64(addr);
          kw[0] = u.x, kw[1] = u.y;
        }
#pragma unroll
        for (int i = 0; i < C::kWords; ++i) {
          uint32_t x[4];
          decode_nibbles(kw[i], x);
          mma_16816(acc, qa[2 * i][0], qa[2 * i][1], qa[2 * i][2], qa[2 * i][3], x[0], x[1]);
          mma_16816(acc, qa[2 * i + 1][0], qa[2 * i + 1][1], qa[2 * i + 1][2], qa[2 * i + 1][3], x[2], x[3]);
        }
        const int j0 = tok0 + nt * 8 + 2 * c, j1 = j0 + 1;
        const float f0 = __half2float(sks[nt * 8 + 2 * c]) * a.scale_log2;
        const float f1 = __half2float(sks[nt * 8 + 2 * c + 1]) * a.scale_log2;
        const bool ok0 = j0 < a.nk, ok1 = j1 < a.nk;
        t[nt][0] = (ok0 && (!a.causal || j0 <= row0 + shift)) ? acc[0] * f0 : -INFINITY;
        t[nt][1] = (ok1 && (!a.causal || j1 <= row0 + shift)) ? acc[1] * f1 : -INFINITY;
        t[nt][2] = (ok0 && (!a.causal || j0 <= row1 + shift)) ? acc[2] * f0 : -INFINITY;
        t[nt][3] = (ok1 && (!a.causal || j1 <= row1 + shift)) ? acc[3] * f1 : -INFINITY;
      }
      float mx0 = t[0][0], mx1 = t[0][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(t[nt][0], t[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(t[nt][2], t[nt][3]));
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      if (n0 > m0 || n1 > m1) {
        const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);
        l0 *= al0, l1 *= al1;
#pragma unroll
        for (int n = 0; n < C::kNt; ++n) o[n][0] *= al0, o[n][1] *= al0, o[n][2] *= al1, o[n][3] *= al1;
        m0 = n0, m1 = n1;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int nt = 2 * kk + h;
          const float p0 = ex2(t[nt][0] - m0), p1 = ex2(t[nt][1] - m0);
          const float p2 = ex2(t[nt][2] - m1), p3 = ex2(t[nt][3] - m1);
          l0 += p0 + p1;
          l1 += p2 + p3;
          const int jl = nt * 8 + 2 * c;
          const float v0 = tok0 + jl < a.nk ? __half2float(svs[jl]) : 0.f;
          const float v1 = tok0 + jl + 1 < a.nk ? __half2float(svs[jl + 1]) : 0.f;
          pa[2 * h] = pack_half2(p0 * v0, p1 * v1);
          pa[2 * h + 1] = pack_half2(p2 * v0, p3 * v1);
        }
        // A regs: a0 = (row g, tok 2c..), a1 = (row g+8, tok 2c..), a2/a3 = tokens +8
#pragma unroll
        for (int jj = 0; jj < D / 64; ++jj) {
          const int q = lane >> 3;
          const int vt = kk * 16 + ((q & 1) ? 8 : 0) + (lane & 7);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_trans(vb + swz128(vt * (D / 2) + (2 * jj + (q >> 1)) * 16), r0, r1, r2, r3);
          uint32_t d0[4], d1[4], d2[4], d3[4];
          decode_nibbles(r0, d0);
          decode_nibbles(r1, d1);
          decode_nibbles(r2, d2);
          decode_nibbles(r3, d3);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            mma_16816(o[(2 * jj) * 4 + e], pa[0], pa[1], pa[2], pa[3], d0[e], d1[e]);
            mma_16816(o[(2 * jj + 1) * 4 + e], pa[0], pa[1], pa[2], pa[3], d2[e], d3[e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }

  // -------------------------------------------------------------- epilogue
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int64_t obase = (static_cast<int64_t>(b) * a.hq + hq) * a.nq;
  __half *out = reinterpret_cast<__half *>(a.out);
#pragma unroll
  for (int j = 0; j < D / 32; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = j * 4 + e, d = 32 * j + 8 * c + e;
      if (row0 < a.nq) {
        out[(obase + row0) * D + d] = __float2half_rn(o[n][0] * inv0);
        out[(obase + row0) * D + d + 4] = __float2half_rn(o[n][1] * inv0);
      }
      if (row1 < a.nq) {
        out[(obase + row1) * D + d] = __float2half_rn(o[n][2] * inv1);
        out[(obase + row1) * D + d + 4] = __float2half_rn(o[n][3] * inv1);
      }
    }
  if (a.lse && c == 0) {
    const float ln2 = 0.69314718055994531f;
    if (row0 < a.nq) a.lse[obase + row0] = l0 > 0.f ? (m0 + log2f(l0)) * ln2 : -INFINITY;
    if (row1 < a.nq) a.lse[obase + row1] = l1 > 0.f ? (m1 + log2f(l1)) * ln2 : -INFINITY;
  }
}

template <int D>
cudaError_t launch_p(const PrefillArgs &a, const KvView &cache, const CUtensorMap &kmap,
                     const CUtensorMap &vmap, uint32_t *err, cudaStream_t stream) {
  using C = PCfg<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid((a.nq + kRows - 1) / kRows, a.hq, a.batch);
  prefill_kernel<D><<<grid, kThreads, C::kSmem, stream>>>(a, cache, kmap, vmap, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, const KvView &cache, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, uint32_t *err, cudaStream_t stream) {
  if (a.batch == 0 || a.nq == 0) return cudaSuccess;
  return cache.head_dim == 128 ? launch_p<128>(a, cache, kmap, vmap, err, stream)
                               : launch_p<64>(a, cache, kmap, vmap, err, stream);
}

}  // namespace qattn
