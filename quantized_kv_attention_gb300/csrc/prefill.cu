// prefill.cu -- prefill attention over the INT4 cache on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// TurboAttention (arXiv 2412.08585) §2.1 (prefill over the cached K, V) and
// §2.2 Eq. 2 with FlashAttention's tiling (Q, K, V chunked along tokens,
// partial attention per pair of chunks, online max and sum, final
// normalisation).  K/V arrive as 4-bit codes plus per-token fp16 scales and
// are dequantized on chip, in shared memory, right ahead of the MMA operand
// stage ("Quantized Cross-Attention ... In-SRAM Dequantization" §3.1); no
// fp16 K/V is ever written to HBM.
//
// One CTA (one per SM) owns two 128-row query tiles that read the same kv
// head: two query heads of one GQA group at the same rows when the group
// size is even, otherwise two consecutive row blocks of one head.  It walks
// the visible keys in tiles of 128:
//   dequant warps (4)   codes of key tile j (plain 16-byte loads) -> exact
//                       fp16 integers in 128B-swizzled K and V operand
//                       tiles (double-buffered); per-token factors
//                       kf = s_K * softmax_scale * log2(e) and vf = s_V
//   MMA thread (1)      S_t = Q_t . codes_K^T   (M=128, N=128, K=D; SMEM x SMEM)
//                       O_t += P_t . codes_V    (M=128, N=D, K=128; P from TMEM)
//   softmax warps (2x4) one thread per query row: x = S*kf - m, p = 2^x,
//                       P = fp16(p * vf) back into TMEM over S; lazy max:
//                       m moves only when a tile's sum exceeds 2^8, then O is
//                       rescaled in TMEM before the next PV
// TMEM: S_0 | S_1 | O_0 | O_1 (512 columns).  The epilogue divides O by the
// row sum, stages it in the Q tile's shared memory and stores it with TMA.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace qattn {
namespace {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // keys per tile
constexpr int kSoftmaxThreads = 256;
constexpr int kDequantThreads = 128;
constexpr int kMmaWarp = 12;        // warpgroup 3; its other three warps idle
constexpr int kThreads = 512;       // four warpgroups: softmax 0, softmax 1, dequant, MMA
// Registers per thread after the split (launch: 128); one warp of every
// warpgroup sits on each SM sub-partition, so the per-partition total stays
// 160 + 160 + 96 + 96 = 512 = 4 x 128.
constexpr int kRegsSoftmax = 160, kRegsDequant = 96, kRegsMma = 96;
constexpr int kKvBufs = 2;
constexpr int kScaleSlots = 4;
constexpr int kRedoSum = 256;  // a tile whose sum of 2^x exceeds this moves the max

template <int D>
struct TcCfg {
  static constexpr int kSub = D / 64;           // 64-column (128-byte) subtiles
  static constexpr int kSubBytes = 128 * 128;   // one subtile of a 128-row tile
  static constexpr int kTileBytes = kSub * kSubBytes;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKvBufs * kTileBytes;
  static constexpr int kScOff = kVOff + kKvBufs * kTileBytes;
  static constexpr int kBarOff = kScOff + kScaleSlots * 2 * kBN * 4;
  static constexpr int kSmem = kBarOff + 256 + 1024;  // barriers + TMEM base, alignment slack
  static constexpr uint32_t kIdescS = idesc_f16(kBM, kBN, false);
  static constexpr uint32_t kIdescPV = idesc_f16(kBM, D, true);
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKvBufs], k_empty[kKvBufs];
  uint64_t v_full[kKvBufs], v_empty[kKvBufs];
  uint64_t s_full[2], p_full[2];
  uint64_t o_full;
  uint64_t sc_full[kScaleSlots], sc_empty[kScaleSlots];
  uint32_t tmem_base;
};

// One (query-tile pair) work item.
struct Work {
  int b, kvh, h[2], r[2], ntiles;
};

__device__ __forceinline__ Work decode_work(const PrefillArgs &a, int hkv) {
  Work w;
  const int G = a.hq / hkv;
  const int nqb = (a.nq + kBM - 1) / kBM;
  const bool pair_heads = (G % 2) == 0;
  const int P = pair_heads ? G / 2 : G;
  const int nslot = pair_heads ? nqb : (nqb + 1) / 2;
  int idx = blockIdx.x;
  const int p = idx % P;
  idx /= P;
  w.kvh = idx % hkv;
  idx /= hkv;
  w.b = idx % a.batch;
  const int slot = nslot - 1 - idx / a.batch;  // row blocks with the most keys first
  if (pair_heads) {
    w.h[0] = w.kvh * G + 2 * p, w.h[1] = w.h[0] + 1;
    w.r[0] = w.r[1] = slot * kBM;
  } else {
    w.h[0] = w.h[1] = w.kvh * G + p;
    w.r[0] = slot * 2 * kBM, w.r[1] = w.r[0] + kBM;
  }
  const int last_row = min(max(w.r[0], w.r[1]) + kBM - 1, a.nq - 1);
  const int kv_end = a.causal ? min(a.nk, last_row + (a.nk - a.nq) + 1) : a.nk;
  w.ntiles = (kv_end + kBN - 1) / kBN;
  return w;
}

// Two signed nibbles of byte `k` of w -> (low, high) as exact fp16 integers.
// The byte is copied into both halves; the low nibble (xor 8) becomes the
// mantissa of 1024 + (c + 8) in the low half, the high nibble the mantissa
// of 1024 + 16 (c + 8) in the high half; one fma with per-half constants
// leaves c in each.
template <int K>
__device__ __forceinline__ uint32_t nibble_pair(uint32_t w) {
  uint32_t t, x;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(w), "n"(K | (4 << 4) | (K << 8) | (4 << 12)));
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(x) : "r"(t), "r"(0x00F0000Fu), "r"(0x64806408u));
  const __half2 mul = __halves2half2(__ushort_as_half(0x3C00), __ushort_as_half(0x2C00));   // 1, 1/16
  const __half2 add = __halves2half2(__ushort_as_half(0xE408), __ushort_as_half(0xD480));   // -1032, -72
  __half2 h = __hfma2(*reinterpret_cast<__half2 *>(&x), mul, add);
  return *reinterpret_cast<uint32_t *>(&h);
}

// 8 codes (one 32-bit word, element order) -> 16 bytes of fp16 at `dst`.
__device__ __forceinline__ void store_word(uint32_t dst, uint32_t w) {
  const uint32_t a = nibble_pair<0>(w), b = nibble_pair<1>(w), c = nibble_pair<2>(w), d = nibble_pair<3>(w);
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Writes one token row (D codes) as fp16 into a 128B-swizzled tile whose
// rows are tokens: subtile d/64, row `tok`, 16-byte chunk (d%64)/8.
template <int D>
__device__ __forceinline__ void store_row(uint32_t tile, int tok, const uint4 (&c)[D / 32]) {
  const uint32_t row = tile + tok * 128;
  const uint32_t x = tok & 7;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const uint32_t words[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = i * 4 + q;  // 8 elements per chunk
      const uint32_t sub = chunk / 8, col = chunk % 8;
      store_word(row + sub * TcCfg<D>::kSubBytes + ((col ^ x) << 4), words[q]);
    }
  }
}

// Multiplies the P chunks already written (c of them) and, when `o_too`,
// the O row by alpha.  Out of line: it runs only when a row maximum moves.
template <int D>
__device__ __noinline__ void rescale_tmem(uint32_t s_tm, uint32_t o_tm, int c, bool o_too, float alpha) {
  tmem_st_wait();
#pragma unroll 1
  for (int c2 = 0; c2 < c; ++c2) {
    uint32_t ph[16];
    tmem_ld16(s_tm + c2 * 16, ph);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<__half2 *>(&ph[i]));
      ph[i] = pack_half2(f.x * alpha, f.y * alpha);
    }
    tmem_st16(s_tm + c2 * 16, ph);
  }
  if (o_too) {
#pragma unroll 1
    for (int c2 = 0; c2 < D / 32; ++c2) {
      uint32_t o[32];
      tmem_ld32(o_tm + c2 * 32, o);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
      tmem_st32(o_tm + c2 * 32, o);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(PrefillArgs a, KvView cache, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap omap, uint32_t *err) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + C::kBarOff);
  float *scales = reinterpret_cast<float *>(smem + C::kScOff);  // [slot][kf 128 | vf 128]
  const uint32_t sbase = smem_u32(smem);

  const Work w = decode_work(a, cache.hkv);
  const int n = w.ntiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int i = 0; i < kKvBufs; ++i) {
      mbar_init(smem_u32(&bars->k_full[i]), kDequantThreads);
      mbar_init(smem_u32(&bars->v_full[i]), kDequantThreads);
      mbar_init(smem_u32(&bars->k_empty[i]), 1);
      mbar_init(smem_u32(&bars->v_empty[i]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->p_full[t]), kSoftmaxThreads / 2);
    }
    mbar_init(smem_u32(&bars->o_full), 1);
    for (int i = 0; i < kScaleSlots; ++i) {
      mbar_init(smem_u32(&bars->sc_full[i]), kDequantThreads);
      mbar_init(smem_u32(&bars->sc_empty[i]), kSoftmaxThreads);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int wg = warp >> 2;

  // Each role sets its register budget inside its own branch, so that the
  // compiler allocates every branch for that budget.
  if (wg == 3) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
    // ------------------------------------------------------------ MMA issue
    if (warp == kMmaWarp && lane == 0) {
      prefetch_tmap(&qmap);
      const uint32_t qf = smem_u32(&bars->q_full);
      mbar_arrive_expect_tx(qf, 2 * C::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d(sbase + C::kQOff + t * C::kTileBytes + s * C::kSubBytes, &qmap, 64 * s, w.r[t],
                      w.b * a.hq + w.h[t], qf);
      bool ok = mbar_wait(qf, 0, err);
      // Descriptors are built once; a start address moves by adding its
      // 16-byte-unit offset to the low field (addresses stay below 256 KB).
      const uint64_t qdesc = sw128_desc(sbase + C::kQOff, 16, 1024);
      const uint64_t kdesc = sw128_desc(sbase + C::kKOff, 16, 1024);
      const uint64_t vdesc = sw128_desc(sbase + C::kVOff, C::kSubBytes, 1024);
      constexpr uint32_t kTile16 = C::kTileBytes >> 4;
      auto issue_s = [&](int t, int j) {
        const uint64_t qa = qdesc + t * kTile16, kb = kdesc + (j % kKvBufs) * kTile16;
        const uint32_t d = tmem + t * kBN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * C::kSubBytes + (kk % 4) * 32) >> 4;
          umma_ss(d, qa + off, kb + off, C::kIdescS, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int j) {
        const uint64_t vb = vdesc + (j % kKvBufs) * kTile16;
        const uint32_t d = tmem + 256 + t * D, p = tmem + t * kBN;
        const uint32_t acc0 = j > 0;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) umma_ts(d, p + kk * 8, vb + kk * (2048 >> 4), C::kIdescPV, kk > 0 ? 1u : acc0);
      };
      if (ok) ok = mbar_wait(smem_u32(&bars->k_full[0]), 0, err);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        tc_commit(smem_u32(&bars->s_full[0]));
        issue_s(1, 0);
        tc_commit(smem_u32(&bars->s_full[1]));
        tc_commit(smem_u32(&bars->k_empty[0]));
      }
      for (int j = 0; ok && j < n; ++j) {
        const int vbuf = j % kKvBufs;
        const uint32_t par = (j / kKvBufs) & 1;
        if (!(ok = mbar_wait(smem_u32(&bars->v_full[vbuf]), par, err))) break;
        if (!(ok = mbar_wait(smem_u32(&bars->p_full[0]), j & 1, err))) break;
        tc_fence_after();
        issue_pv(0, j);
        const bool more = j + 1 < n;
        if (more) {
          const int kb = (j + 1) % kKvBufs;
          if (!(ok = mbar_wait(smem_u32(&bars->k_full[kb]), ((j + 1) / kKvBufs) & 1, err))) break;
          tc_fence_after();
          issue_s(0, j + 1);
          tc_commit(smem_u32(&bars->s_full[0]));
        }
        if (!(ok = mbar_wait(smem_u32(&bars->p_full[1]), j & 1, err))) break;
        tc_fence_after();
        issue_pv(1, j);
        tc_commit(smem_u32(&bars->v_empty[vbuf]));
        if (more) {
          issue_s(1, j + 1);
          tc_commit(smem_u32(&bars->s_full[1]));
          tc_commit(smem_u32(&bars->k_empty[(j + 1) % kKvBufs]));
        }
      }
      // Always signal o_full so waiters end; then let every MMA finish
      // before the tensor memory is released.
      tc_commit(smem_u32(&bars->o_full));
      mbar_wait(smem_u32(&bars->o_full), 0, err, ok ? kWaitCycles : kDrainCycles);
    }
    __syncwarp();
  } else if (wg == 2) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDequant));
    // ---------------------------------------------------- dequantization
    const int tok_l = threadIdx.x - kSoftmaxThreads;  // token within the tile
    const int64_t row0 = (static_cast<int64_t>(w.b) * cache.hkv + w.kvh) * cache.capacity;
    const uint4 *kc = reinterpret_cast<const uint4 *>(cache.k_codes + row0 * (D / 2));
    const uint4 *vc = reinterpret_cast<const uint4 *>(cache.v_codes + row0 * (D / 2));
    const __half *ks = reinterpret_cast<const __half *>(cache.k_scales) + row0;
    const __half *vs = reinterpret_cast<const __half *>(cache.v_scales) + row0;
    // No prefetch across tiles: the two operand buffers let this warpgroup
    // run up to two tiles ahead of the tensor core, which hides the load.
    for (int j = 0; j < n; ++j) {
      const int tok = j * kBN + tok_l;
      uint4 ck[D / 32], cv[D / 32];
      float fk = 0.f, fv = 0.f;
      if (tok < a.nk) {
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          ck[i] = __ldg(kc + static_cast<int64_t>(tok) * (D / 32) + i);
          cv[i] = __ldg(vc + static_cast<int64_t>(tok) * (D / 32) + i);
        }
        fk = __half2float(ks[tok]) * a.scale_log2;
        fv = __half2float(vs[tok]);
      } else {
#pragma unroll
        for (int i = 0; i < D / 32; ++i) ck[i] = cv[i] = make_uint4(0, 0, 0, 0);
      }
      const int buf = j % kKvBufs;
      const uint32_t par = ((j / kKvBufs) & 1) ^ 1;
      if (j >= kKvBufs && !mbar_wait(smem_u32(&bars->k_empty[buf]), par, err)) break;
      store_row<D>(sbase + C::kKOff + buf * C::kTileBytes, tok_l, ck);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars->k_full[buf]));
      const int slot = j % kScaleSlots;
      if (j >= kScaleSlots &&
          !mbar_wait(smem_u32(&bars->sc_empty[slot]), ((j / kScaleSlots) & 1) ^ 1, err))
        break;
      scales[slot * 2 * kBN + tok_l] = fk;
      scales[slot * 2 * kBN + kBN + tok_l] = fv;
      mbar_arrive(smem_u32(&bars->sc_full[slot]));
      if (j >= kKvBufs && !mbar_wait(smem_u32(&bars->v_empty[buf]), par, err)) break;
      store_row<D>(sbase + C::kVOff + buf * C::kTileBytes, tok_l, cv);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars->v_full[buf]));
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2, wq = warp & 3;
    const int row_l = wq * 32 + lane;
    const int row = w.r[t] + row_l;
    const int shift = a.nk - a.nq;
    const int limit = a.causal ? min(a.nk - 1, row + shift) : a.nk - 1;  // last visible key
    const int warp_limit = a.causal ? min(a.nk - 1, w.r[t] + wq * 32 + shift) : a.nk - 1;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + t * kBN;
    const uint32_t o_tm = tmem + lane_off + 256 + t * D;
    float m = 0.f, l = 0.f;
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      const int slot = j % kScaleSlots;
      if (!(ok = mbar_wait(smem_u32(&bars->sc_full[slot]), (j / kScaleSlots) & 1, err))) break;
      if (!(ok = mbar_wait(smem_u32(&bars->s_full[t]), j & 1, err))) break;
      tc_fence_after();
      const float *kf = scales + slot * 2 * kBN;
      const float *vf = kf + kBN;
      const int key0 = j * kBN;
      const bool masked = key0 + kBN - 1 > warp_limit;

      // maximum of S*kf over one 32-key chunk (masked keys excluded)
      auto chunk_max = [&](const uint32_t(&s)[32], int c) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 f = *reinterpret_cast<const float4 *>(kf + c * 32 + i);
          const float fs[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x = __uint_as_float(s[i + e]) * fs[e];
            mx = fmaxf(mx, (masked && key0 + c * 32 + i + e > limit) ? -INFINITY : x);
          }
        }
        return mx;
      };
      // p = 2^(S*kf - m) of one chunk; h = fp16 pairs of p*vf; returns the sum of p
      auto chunk_exp = [&](const uint32_t(&s)[32], int c, uint32_t(&h)[16]) {
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 f = *reinterpret_cast<const float4 *>(kf + c * 32 + i);
          const float4 g = *reinterpret_cast<const float4 *>(vf + c * 32 + i);
          const float fs[4] = {f.x, f.y, f.z, f.w}, gs[4] = {g.x, g.y, g.z, g.w};
          float p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = fmaf(__uint_as_float(s[i + e]), fs[e], -m);
            if (masked && key0 + c * 32 + i + e > limit) x = -INFINITY;
            p[e] = ex2(x);
          }
          sum0 += p[0] + p[2], sum1 += p[1] + p[3];
          h[i / 2] = pack_half2(p[0] * gs[0], p[1] * gs[1]);
          h[i / 2 + 1] = pack_half2(p[2] * gs[2], p[3] * gs[3]);
        }
        return sum0 + sum1;
      };

      if (j == 0) {  // the first tile fixes the reference maximum
        float mx = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t s[32];
          tmem_ld32(s_tm + c * 32, s);
          mx = fmaxf(mx, chunk_max(s, c));
        }
        m = mx == -INFINITY ? 0.f : mx;
      }
      // P chunk c (16 columns) overwrites S columns already read.
      float tsum = 0.f;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t s[32], h[16];
        tmem_ld32(s_tm + c * 32, s);
        float cs = chunk_exp(s, c, h);
        if (__any_sync(0xffffffffu, !(cs <= static_cast<float>(kRedoSum)))) {
          // the reference maximum moves: rescale what was built on the old one
          const float mn = fmaxf(m, chunk_max(s, c));
          const float alpha = ex2(m - mn);
          m = mn, l *= alpha, tsum *= alpha;
          rescale_tmem<D>(s_tm, o_tm, c, j > 0, alpha);
          tmem_ld32(s_tm + c * 32, s);  // S chunk c is intact: P so far only covers chunks < c/2
          cs = chunk_exp(s, c, h);
        }
        tsum += cs;
        tmem_st16(s_tm + c * 16, h);
      }
      l += tsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full[t]));
      mbar_arrive(smem_u32(&bars->sc_empty[slot]));
    }

    // ------------------------------------------------------------ epilogue
    const bool done = mbar_wait(smem_u32(&bars->o_full), 0, err, ok ? kWaitCycles : kDrainCycles);
    tc_fence_after();
    if (done && ok) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint32_t stage = sbase + C::kQOff + t * C::kTileBytes;  // Q tile t is no longer read
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(o_tm + c * 32, o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = c * 4 + q;
          const uint32_t sub = chunk / 8, col = chunk % 8;
          const uint32_t h0 = pack_half2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          const uint32_t h1 = pack_half2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          const uint32_t h2 = pack_half2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          const uint32_t h3 = pack_half2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
          const uint32_t dst = stage + sub * C::kSubBytes + row_l * 128 + ((col ^ (row_l & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(h0), "r"(h1), "r"(h2), "r"(h3)
                       : "memory");
        }
      }
      // each warp stores its own 32 rows (no cross-warp barrier)
      fence_proxy_async_smem();
      __syncwarp();
      const int wrow = w.r[t] + wq * 32;
      if (lane == 0 && wrow < a.nq) {
        for (int s = 0; s < C::kSub; ++s)
          tma_store_3d(&omap, stage + s * C::kSubBytes + wq * 32 * 128, 64 * s, wrow, w.b * a.hq + w.h[t]);
        bulk_commit_group();
        bulk_wait_read_all();
      }
      if (a.lse && row < a.nq) {
        const int64_t li = (static_cast<int64_t>(w.b) * a.hq + w.h[t]) * a.nq + row;
        a.lse[li] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_tc(const PrefillArgs &a, const KvView &cache, const CUtensorMap &qmap,
                      const CUtensorMap &omap, uint32_t *err, cudaStream_t stream) {
  using C = TcCfg<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int G = a.hq / cache.hkv;
  const int nqb = (a.nq + kBM - 1) / kBM;
  const int64_t items = (G % 2 == 0) ? static_cast<int64_t>(a.batch) * cache.hkv * (G / 2) * nqb
                                     : static_cast<int64_t>(a.batch) * a.hq * ((nqb + 1) / 2);
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_tc_kernel<D><<<static_cast<unsigned>(items), kThreads, C::kSmem, stream>>>(a, cache, qmap, omap, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, const KvView &cache, const CUtensorMap &qmap,
                           const CUtensorMap &omap, uint32_t *err, cudaStream_t stream) {
  if (a.batch == 0 || a.nq == 0) return cudaSuccess;
  return cache.head_dim == 128 ? launch_tc<128>(a, cache, qmap, omap, err, stream)
                               : launch_tc<64>(a, cache, qmap, omap, err, stream);
}

}  // namespace qattn
