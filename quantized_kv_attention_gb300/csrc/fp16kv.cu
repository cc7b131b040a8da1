// fp16kv.cu -- the comparison paths of "Quantized Cross-Attention ... In-SRAM
// Dequantization", §5.2 (Baselines): attention over an FP16 KV cache (the
// page's FP16 FlashAttention-3 arm), and post-dequantization, where the INT4
// cache is first written back to HBM as FP16 (dequantize_kernel) and that
// copy is then attended by the same FP16 kernels.  They exist to measure on
// this GPU what the fused kernels save; they follow the fused kernels'
// conventions (GQA, split-KV with a log-sum-exp merge).
//
// decode16_kernel: one CTA per (key split, sequence, kv-head), tokens on M of
// mma.sync m16n8k16 and the G query heads of the kv-head on N, as in the INT4
// decode.  A producer thread streams 64-token K and V tiles by TMA (128-byte
// swizzle) into a 6-deep ring (12 at D = 64); 4 consumer warps take 16
// tokens of each tile: S^T = K . Q^T (K by ldmatrix), online softmax in the
// log2 domain with a lazy maximum, O^T += V^T . P^T (V by ldmatrix.trans, P
// moved to the B layout by movmatrix).  The warps merge in shared memory;
// with one split the CTA writes O and lse, else an fp32 partial that the
// combine kernel merges.
#include <math.h>

#include "../../include/qattn.h"
#include "internal.h"
#include "ptx.cuh"

namespace qattn {
namespace {

// ---------------------------------------------------------------- dequantize
// x16 = fl16(c * s): decode_nibbles gives the exact fp16 codes, the permutes
// restore element order, and HMUL2 of two fp16 values is the correctly
// rounded product.  One thread per 8 codes (one 32-bit word) of a row: a
// warp reads 128 contiguous bytes of codes and writes 512 contiguous bytes.
__device__ __forceinline__ uint4 dequant_word_pairs(uint32_t w, __half2 s2) {
  uint32_t x[4];
  decode_nibbles(w, x);  // (e0, e4), (e1, e5), (e2, e6), (e3, e7)
  const uint32_t p[4] = {__byte_perm(x[0], x[1], 0x5410), __byte_perm(x[2], x[3], 0x5410),
                         __byte_perm(x[0], x[1], 0x7632), __byte_perm(x[2], x[3], 0x7632)};
  uint32_t r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 y = __hmul2(*reinterpret_cast<const __half2 *>(&p[k]), s2);
    r[k] = *reinterpret_cast<const uint32_t *>(&y);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

template <int D>
__global__ void __launch_bounds__(256)
    dequantize_kernel(KvView cache, int batch, int n, uint16_t *__restrict__ k_out, uint16_t *__restrict__ v_out,
                      uint32_t *err) {
  constexpr int WPR = D / 8;  // 32-bit code words per row; a thread turns one into 16 bytes of fp16
  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;
  const int64_t total = rows * WPR;
  const bool small = rows <= 0x7fffffffLL;  // row / n in 32 bits
  const bool is_v = blockIdx.y != 0;
  const uint32_t *codes = reinterpret_cast<const uint32_t *>(is_v ? cache.v_codes : cache.k_codes);
  const uint16_t *scales = is_v ? cache.v_scales : cache.k_scales;
  uint4 *out = reinterpret_cast<uint4 *>(is_v ? v_out : k_out);
  // four words a thread per pass (the grid's stride apart), their loads issued together
  constexpr int U = 4;
  auto src_row = [&](int64_t row) -> int64_t {
    int64_t bh;
    int i;
    if (small) {
      const uint32_t r32 = static_cast<uint32_t>(row), q = r32 / static_cast<uint32_t>(n);
      bh = q, i = static_cast<int>(r32 - q * static_cast<uint32_t>(n));
    } else {
      bh = row / n, i = static_cast<int>(row - bh * n);
    }
    if (cache.page_table == nullptr) return bh * cache.capacity + i;
    const int h = static_cast<int>(bh % cache.hkv), b = static_cast<int>(bh / cache.hkv);
    const int page = __ldg(cache.page_table + static_cast<int64_t>(b) * cache.max_pages + i / kPage);
    if (page >= 0 && page < cache.num_pages) return (static_cast<int64_t>(page) * cache.hkv + h) * kPage + i % kPage;
    return -1;
  };
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t0 < total; t0 += U * stride) {
    uint32_t c[U];
    uint16_t sc[U];
    int64_t src[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = t0 + u * stride;
      src[u] = t < total ? src_row(t / WPR) : -2;
      if (src[u] == -1 && t % WPR == 0) atomicOr(err, kFlagBadPage);
      c[u] = src[u] >= 0 ? __ldg(codes + src[u] * WPR + static_cast<int>(t % WPR)) : 0u;
      sc[u] = src[u] >= 0 ? __ldg(scales + src[u]) : static_cast<uint16_t>(0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = t0 + u * stride;
      if (src[u] == -2) break;
      out[t] = src[u] >= 0 ? dequant_word_pairs(c[u], __half2half2(__ushort_as_half(sc[u]))) : make_uint4(0, 0, 0, 0);
    }
  }
}

// ------------------------------------------------------------- fp16 decode
constexpr int kW16 = 4;            // consumer warps, 16 tokens of each tile
constexpr int kT16 = 16 * kW16;    // tokens per tile
constexpr int kThreads16 = (kW16 + 1) * 32;

template <int D>
struct C16 {
  static constexpr int kSub = D / 64;                  // 64-column (128-byte) subtiles
  static constexpr int kSubBytes = kT16 * 128;         // 8 KB
  static constexpr int kTile = kSub * kSubBytes;       // K or V of one stage
  static constexpr int kStageBytes = 2 * kTile;
  static constexpr int kStages = D == 128 ? 6 : 12;
  static constexpr int kPitch = D + 4;                 // fp32 merge row pitch
  static constexpr int kMergeBytes = kW16 * 8 * kPitch * 4;
  static constexpr int kSmem = kStages * kStageBytes + kMergeBytes + 2 * kW16 * 8 * 4 + 2 * kStages * 8 + 16 + 1024;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Shared-memory address of 16-byte chunk `chunk` (8 fp16 along D) of token
// row `tok` in a TMA tile of kSub subtiles written with the 128-byte swizzle.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int tok, int chunk) {
  return tile + (chunk >> 3) * C16<D>::kSubBytes + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kThreads16, 1)
    decode16_kernel(const uint16_t *__restrict__ q, const int32_t *__restrict__ seq_lens, int batch, int hq,
                    int hkv, int64_t capacity, int chunk, float scale_log2, uint16_t *__restrict__ out,
                    float *__restrict__ lse, float *__restrict__ partial_o, float *__restrict__ partial_lse,
                    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    uint32_t *err) {
  using C = C16<D>;
  constexpr int kMt = D / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *mo = reinterpret_cast<float *>(smem + C::kStages * C::kStageBytes);  // [warp][head][kPitch]
  float *mm = mo + kW16 * 8 * C::kPitch;                                      // [warp][head]
  float *ml = mm + kW16 * 8;
  uint64_t *full = reinterpret_cast<uint64_t *>(ml + kW16 * 8);
  uint64_t *empty = full + C::kStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, splits = gridDim.x;
  const int bh = blockIdx.y, b = bh / hkv, kvh = bh % hkv;
  const int G = hq / hkv;
  const int64_t len = min(static_cast<int64_t>(max(__ldg(seq_lens + b), 0)), capacity);
  const int64_t t0 = static_cast<int64_t>(split) * chunk;
  const int64_t t1 = min(t0 + chunk, len);
  const int nst = t1 > t0 ? static_cast<int>((t1 - t0 + kT16 - 1) / kT16) : 0;
  const int64_t row0 = static_cast<int64_t>(b) * hq + static_cast<int64_t>(kvh) * G;  // first q-head row

  if (nst == 0) {  // no key in this split: an empty partial (or, unsplit, O = 0)
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      if (splits == 1) out[row0 * D + i] = 0;
      if (i % D == 0) {
        const int64_t r = row0 + i / D;
        if (splits == 1) {
          if (lse) lse[r] = -INFINITY;
        } else {
          partial_lse[static_cast<int64_t>(split) * batch * hq + r] = -INFINITY;
        }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kW16);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kW16) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      for (int j = 0; j < nst; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages &&
            !mbar_wait(smem_u32(empty + s), ((j / C::kStages) & 1) ^ 1, err, *abort_flag ? kDrainCycles : kWaitCycles)) {
          *abort_flag = 1;
          break;
        }
        const uint32_t st = smem_u32(smem + s * C::kStageBytes);
        const uint32_t bar = smem_u32(full + s);
        const int tok = static_cast<int>(t0) + j * kT16;
        mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
        for (int sub = 0; sub < C::kSub; ++sub) {
          tma_load_3d(st + sub * C::kSubBytes, &kmap, 64 * sub, tok, bh, bar);
          tma_load_3d(st + C::kTile + sub * C::kSubBytes, &vmap, 64 * sub, tok, bh, bar);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  // Q^T as the B operand: k-step kk covers d = 16 kk .. 16 kk + 15, column g
  // is q-head g of the group (zero past G)
  uint32_t qb[kMt][2];
  {
    const uint32_t *qr = reinterpret_cast<const uint32_t *>(q + (row0 + min(g, G - 1)) * D);
#pragma unroll
    for (int kk = 0; kk < kMt; ++kk) {
      qb[kk][0] = g < G ? __ldg(qr + 8 * kk + c) : 0u;
      qb[kk][1] = g < G ? __ldg(qr + 8 * kk + 4 + c) : 0u;
    }
  }
  float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f;
  float o[kMt][4];
#pragma unroll
  for (int mt = 0; mt < kMt; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  // ldmatrix row addresses: K (matrix q = lane / 8: tokens (q & 1) * 8 + 0..7,
  // chunk 2 kk + q / 2); V transposed (tokens (q / 2) * 8 + 0..7, chunk 2 mt + (q & 1))
  const int mq = lane >> 3;
  const int ktok = warp * 16 + (lane & 7) + (mq & 1) * 8, kch = mq >> 1;
  const int vtok = warp * 16 + (lane & 7) + (mq >> 1) * 8, vch = mq & 1;

  for (int j = 0; j < nst; ++j) {
    const int s = j % C::kStages;
    const bool got = mbar_wait(smem_u32(full + s), (j / C::kStages) & 1, err, *abort_flag ? kDrainCycles : kWaitCycles);
    if (!got) *abort_flag = 1;
    const int64_t tok0 = t0 + static_cast<int64_t>(j) * kT16 + warp * 16;
    const int nvalid = got ? static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(16), t1 - tok0))) : 0;
    if (nvalid > 0) {
      const uint32_t kt = smem_u32(smem + s * C::kStageBytes), vt = kt + C::kTile;
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < kMt; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(tile_addr<D>(kt, ktok, 2 * kk + kch), a0, a1, a2, a3);
        if (kk & 1)
          mma_16816(sb, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        else
          mma_16816(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
      // scores (log2 units) of tokens g, g + 8 for q-heads 2c, 2c + 1
      float ts0 = (sa[0] + sb[0]) * scale_log2, ts1 = (sa[1] + sb[1]) * scale_log2;
      float ts2 = (sa[2] + sb[2]) * scale_log2, ts3 = (sa[3] + sb[3]) * scale_log2;
      if (g >= nvalid) ts0 = ts1 = -INFINITY;
      if (g + 8 >= nvalid) ts2 = ts3 = -INFINITY;
      const float lm0 = fmaxf(ts0, ts2), lm1 = fmaxf(ts1, ts3);
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
        l0 *= al0, l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < kMt; ++mt) o[mt][0] *= al0, o[mt][1] *= al1, o[mt][2] *= al0, o[mt][3] *= al1;
      }
      const float p0 = ex2(ts0 - m0), p1 = ex2(ts1 - m1), p2 = ex2(ts2 - m0), p3 = ex2(ts3 - m1);
      const uint32_t r0 = pack_half2(p0, p1), r1 = pack_half2(p2, p3);
      {  // the sum of the fp16 P the MMA multiplies
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&r0));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&r1));
        l0 += f0.x + f1.x, l1 += f0.y + f1.y;
      }
      const uint32_t pb0 = movmatrix_trans(r0), pb1 = movmatrix_trans(r1);
      // a tail tile's V rows past the keys may hold anything: zero them
      const uint32_t keep01 = (2 * c < nvalid ? 0x0000FFFFu : 0u) | (2 * c + 1 < nvalid ? 0xFFFF0000u : 0u);
      const uint32_t keep23 = (2 * c + 8 < nvalid ? 0x0000FFFFu : 0u) | (2 * c + 9 < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(tile_addr<D>(vt, vtok, 2 * mt + vch), a0, a1, a2, a3);
        if (nvalid < 16) a0 &= keep01, a1 &= keep01, a2 &= keep23, a3 &= keep23;
        mma_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }

  // ----------------------------------------------------- merge the 4 warps
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  float *mw = mo + warp * 8 * C::kPitch;
#pragma unroll
  for (int mt = 0; mt < kMt; ++mt) {
    mw[(2 * c) * C::kPitch + 16 * mt + g] = o[mt][0];
    mw[(2 * c + 1) * C::kPitch + 16 * mt + g] = o[mt][1];
    mw[(2 * c) * C::kPitch + 16 * mt + g + 8] = o[mt][2];
    mw[(2 * c + 1) * C::kPitch + 16 * mt + g + 8] = o[mt][3];
  }
  if (g == 0) {
    mm[warp * 8 + 2 * c] = m0, mm[warp * 8 + 2 * c + 1] = m1;
    ml[warp * 8 + 2 * c] = l0, ml[warp * 8 + 2 * c + 1] = l1;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kW16 * 32) : "memory");
  for (int i = threadIdx.x; i < G * D; i += kW16 * 32) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW16; ++w)
      if (ml[w * 8 + h] > 0.f) M = fmaxf(M, mm[w * 8 + h]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kW16; ++w) {
        if (!(ml[w * 8 + h] > 0.f)) continue;
        const float f = ex2(mm[w * 8 + h] - M);
        L += ml[w * 8 + h] * f;
        acc += mo[(w * 8 + h) * C::kPitch + d] * f;
      }
    }
    const bool live = L > 0.f;
    const float ov = live ? acc / L : 0.f;
    const float lv = live ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    const int64_t r = row0 + h;
    if (splits == 1) {
      out[r * D + d] = __half_as_ushort(__float2half_rn(ov));
      if (d == 0 && lse) lse[r] = lv;
    } else {
      const int64_t pr = static_cast<int64_t>(split) * batch * hq + r;
      partial_o[pr * D + d] = ov;
      if (d == 0) partial_lse[pr] = lv;
    }
  }
}

template <int D>
cudaError_t launch_decode16_t(const Decode16Args &a, const CUtensorMap &kmap, const CUtensorMap &vmap, uint32_t *err,
                              cudaStream_t stream) {
  using C = C16<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(a.splits, a.batch * a.hkv);
  float *po = a.splits > 1 ? a.partial_o : nullptr;
  float *pl = a.splits > 1 ? a.partial_lse : nullptr;
  decode16_kernel<D><<<grid, kThreads16, C::kSmem, stream>>>(a.q, a.seq_lens, a.batch, a.hq, a.hkv, a.capacity,
                                                             a.chunk, a.scale_log2, a.out, a.lse, po, pl, kmap, vmap,
                                                             err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  return launch_combine(a.partial_o, a.partial_lse, a.splits, static_cast<int64_t>(a.batch) * a.hq, D, a.out, a.lse,
                        false, stream);
}

}  // namespace

cudaError_t launch_dequantize(const KvView &cache, int batch, int n, uint16_t *k_out, uint16_t *v_out, uint32_t *err,
                              int sms, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;
  if (rows == 0) return cudaSuccess;
  const int64_t threads = rows * (cache.head_dim / 8);
  const int64_t blocks = min((threads + 255) / 256, static_cast<int64_t>(16) * (sms > 0 ? sms : 1));
  dim3 grid(static_cast<unsigned>(blocks), 2);
  if (cache.head_dim == 128)
    dequantize_kernel<128><<<grid, 256, 0, stream>>>(cache, batch, n, k_out, v_out, err);
  else
    dequantize_kernel<64><<<grid, 256, 0, stream>>>(cache, batch, n, k_out, v_out, err);
  return cudaGetLastError();
}

cudaError_t launch_decode16(const Decode16Args &a, const CUtensorMap &kmap, const CUtensorMap &vmap, uint32_t *err,
                            cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_decode16_t<128>(a, kmap, vmap, err, stream)
                           : launch_decode16_t<64>(a, kmap, vmap, err, stream);
}

}  // namespace qattn
