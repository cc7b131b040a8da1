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
//   dequant warps (4)   codes of key tile j (plain 16-byte loads) -> K as
//                       exact fp16 integers, V as fp16 code * s_V, in
//                       128B-swizzled operand tiles (double-buffered); per-
//                       token factors kf = s_K * softmax_scale * log2(e)
//   MMA thread (1)      S_t = Q_t . codes_K^T   (M=128, N=128, K=D; SMEM x SMEM)
//                       O_t += P_t . V          (M=128, N=D, K=128; P from TMEM)
//   softmax warps (2x4) one thread per query row: x = S*kf - m, p = 2^x,
//                       P = fp16(p) back into TMEM over S; lazy max:
//                       m moves only when a 32-key chunk's sum exceeds 2^8,
//                       then P so far and O are rescaled in TMEM
// TMEM: S_0 | S_1 | O_0 | O_1 (512 columns).  The epilogue divides O by the
// row sum, stages it in the Q tile's shared memory and stores it with TMA.
// Codes unpack to fp16 in the order d0 d4 d1 d5 d2 d6 d3 d7 inside every
// group of 8 columns (the cheapest unpack); warpgroup 3 permutes Q the same
// way once per CTA and the epilogue restores the order of O.
#include <math.h>

#include <type_traits>

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
  static constexpr int kBarOff = kScOff + kScaleSlots * kBN * 4;
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

// Bounded mbarrier wait; the clock is read once every 32 polls so that a
// waiting warp takes few issue slots from the working ones.  kHinted polls
// pass a 32 ns suspend-time hint: the MMA thread and the dequantization
// warps resume sooner after the phase completes (about 1 % of the prefill);
// the softmax warps keep the default suspension, which measured faster for
// them.
template <bool kHinted = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint32_t *err,
                                           long long limit = kWaitCycles) {
  auto poll = [&] { return kHinted ? mbar_try_wait_sleep(bar, parity, 32) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (poll()) return true;
    if ((it & 31u) == 0 && clock64() - t0 > limit) {
      atomicOr(err, kFlagWaitTimeout);
      return false;
    }
  }
}

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

// 8 codes (one 32-bit word) -> 16 bytes of fp16 at `dst`, in the order
// d0 d4 d1 d5 d2 d6 d3 d7 that decode_nibbles yields; when SCALED each code
// is multiplied by the token's scale s2 (one rounding of code * scale).  Q is
// permuted the same way inside every 8-column group (the contraction over d
// does not see it) and the epilogue undoes it on O.
template <bool SCALED>
__device__ __forceinline__ void store_word(uint32_t dst, uint32_t w, __half2 s2) {
  uint32_t x[4];
  decode_nibbles(w, x);
  if (SCALED) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 y = __hmul2(*reinterpret_cast<__half2 *>(&x[k]), s2);
      x[k] = *reinterpret_cast<const uint32_t *>(&y);
    }
  }
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3])
               : "memory");
}

// Writes one token row (D codes, times s2 when SCALED) as fp16 into a
// 128B-swizzled tile whose rows are tokens: subtile d/64, row `tok`, 16-byte
// chunk (d%64)/8.
template <int D, bool SCALED>
__device__ __forceinline__ void store_row(uint32_t tile, int tok, const uint4 (&c)[D / 32], __half2 s2) {
  const uint32_t row = tile + tok * 128;
  const uint32_t x = tok & 7;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const uint32_t words[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = i * 4 + q;  // 8 elements per chunk
      const uint32_t sub = chunk / 8, col = chunk % 8;
      store_word<SCALED>(row + sub * TcCfg<D>::kSubBytes + ((col ^ x) << 4), words[q], s2);
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

// Maximum of S * kf over one 32-key chunk; keys above `limit` are excluded
// when MASK.  kf: shared address of the chunk's 32 factors; k0: its first key.
template <bool MASK>
__device__ __forceinline__ float chunk_max(const uint32_t (&s)[32], uint32_t kf, int k0, int limit) {
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const uint4 f = lds128(kf + i * 4);
    float2 x01 = f2_split(mul2(f2(__uint_as_float(s[i]), __uint_as_float(s[i + 1])),
                               f2(__uint_as_float(f.x), __uint_as_float(f.y))));
    float2 x23 = f2_split(mul2(f2(__uint_as_float(s[i + 2]), __uint_as_float(s[i + 3])),
                               f2(__uint_as_float(f.z), __uint_as_float(f.w))));
    if (MASK) {
      if (k0 + i > limit) x01.x = -INFINITY;
      if (k0 + i + 1 > limit) x01.y = -INFINITY;
      if (k0 + i + 2 > limit) x23.x = -INFINITY;
      if (k0 + i + 3 > limit) x23.y = -INFINITY;
    }
    mx = fmax3(mx, x01.x, x01.y);
    mx = fmax3(mx, x23.x, x23.y);
  }
  return mx;
}

// p = 2^(S * kf - m) over one chunk, lanes paired in f32x2 arithmetic; h gets
// the fp16 pairs of p (the P operand); returns the sum of p.
template <bool MASK>
__device__ __forceinline__ float chunk_exp(const uint32_t (&s)[32], uint32_t kf, float m, int k0, int limit,
                                           uint32_t (&h)[16]) {
  const uint64_t nm = f2(-m, -m);
  uint64_t acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const uint4 f = lds128(kf + i * 4);
    float2 x01 = f2_split(fma2(f2(__uint_as_float(s[i]), __uint_as_float(s[i + 1])),
                               f2(__uint_as_float(f.x), __uint_as_float(f.y)), nm));
    float2 x23 = f2_split(fma2(f2(__uint_as_float(s[i + 2]), __uint_as_float(s[i + 3])),
                               f2(__uint_as_float(f.z), __uint_as_float(f.w)), nm));
    if (MASK) {
      if (k0 + i > limit) x01.x = -INFINITY;
      if (k0 + i + 1 > limit) x01.y = -INFINITY;
      if (k0 + i + 2 > limit) x23.x = -INFINITY;
      if (k0 + i + 3 > limit) x23.y = -INFINITY;
    }
    const float p0 = ex2(x01.x), p1 = ex2(x01.y), p2 = ex2(x23.x), p3 = ex2(x23.y);
    acc0 = add2(acc0, f2(p0, p1)), acc1 = add2(acc1, f2(p2, p3));
    h[i / 2] = pack_half2(p0, p1);
    h[i / 2 + 1] = pack_half2(p2, p3);
  }
  const float2 t2 = f2_split(add2(acc0, acc1));
  return t2.x + t2.y;
}

// KV16: K and V come from an fp16 cache (the comparison path of "Quantized
// Cross-Attention ... In-SRAM Dequantization" §5.2) through kmap / vmap (3-D
// [batch*Hkv][nk][D], 128B swizzle, boxes of 64 columns x 128 keys): one
// thread of warpgroup 2 loads each tile by TMA into the same swizzled operand
// layout the dequantization writes, the per-key factor is the softmax scale,
// and Q and O keep the natural column order.
template <int D, bool KV16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(PrefillArgs a, KvView cache, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, uint32_t *err) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + C::kBarOff);
  float *scales = reinterpret_cast<float *>(smem + C::kScOff);  // [slot][kf of 128 keys]
  const uint32_t sbase = smem_u32(smem);

  const Work w = decode_work(a, cache.hkv);
  const int n = w.ntiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int i = 0; i < kKvBufs; ++i) {
      mbar_init(smem_u32(&bars->k_full[i]), KV16 ? 1 : kDequantThreads);
      mbar_init(smem_u32(&bars->v_full[i]), KV16 ? 1 : kDequantThreads);
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
    const uint32_t qf = smem_u32(&bars->q_full);
    if (warp == kMmaWarp && lane == 0) {
      prefetch_tmap(&qmap);
      mbar_arrive_expect_tx(qf, 2 * C::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d(sbase + C::kQOff + t * C::kTileBytes + s * C::kSubBytes, &qmap, 64 * s, w.r[t],
                      w.b * a.hq + w.h[t], qf);
    }
    // Q columns into the K operand's order (d0 d4 d1 d5 d2 d6 d3 d7 per group of 8)
    const bool qok = wait_bounded(qf, 0, err);
    if (qok && !KV16) {
      for (int ch = threadIdx.x - 3 * 128; ch < 2 * C::kTileBytes / 16; ch += 128) {
        const uint32_t addr = sbase + C::kQOff + ch * 16;
        uint4 v = lds128(addr);
        uint32_t n0, n1, n2, n3;
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(n0) : "r"(v.x), "r"(v.z));
        asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(n1) : "r"(v.x), "r"(v.z));
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(n2) : "r"(v.y), "r"(v.w));
        asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(n3) : "r"(v.y), "r"(v.w));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(n0), "r"(n1), "r"(n2), "r"(n3)
                     : "memory");
      }
      fence_proxy_async_smem();
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp == kMmaWarp && lane == 0) {
      bool ok = qok;
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
      if (ok) ok = wait_bounded<true>(smem_u32(&bars->k_full[0]), 0, err);
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
        if (!(ok = wait_bounded<true>(smem_u32(&bars->v_full[vbuf]), par, err))) break;
        if (!(ok = wait_bounded<true>(smem_u32(&bars->p_full[0]), j & 1, err))) break;
        tc_fence_after();
        issue_pv(0, j);
        const bool more = j + 1 < n;
        if (more) {
          const int kb = (j + 1) % kKvBufs;
          if (!(ok = wait_bounded<true>(smem_u32(&bars->k_full[kb]), ((j + 1) / kKvBufs) & 1, err))) break;
          tc_fence_after();
          issue_s(0, j + 1);
          tc_commit(smem_u32(&bars->s_full[0]));
        }
        if (!(ok = wait_bounded<true>(smem_u32(&bars->p_full[1]), j & 1, err))) break;
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
      wait_bounded(smem_u32(&bars->o_full), 0, err, ok ? kWaitCycles : kDrainCycles);
    }
    __syncwarp();
  } else if (wg == 2) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDequant));
    // ---------------------------------------------------- dequantization
    const int tok_l = threadIdx.x - kSoftmaxThreads;  // token within the tile
    if constexpr (KV16) {
      const int64_t head = static_cast<int64_t>(w.b) * cache.hkv + w.kvh;
      if (tok_l == 0) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
      }
      for (int j = 0; j < n; ++j) {
        const int buf = j % kKvBufs;
        const uint32_t par = ((j / kKvBufs) & 1) ^ 1;
        if (tok_l == 0) {
          if (j >= kKvBufs && !wait_bounded<true>(smem_u32(&bars->k_empty[buf]), par, err)) break;
          const uint32_t kf = smem_u32(&bars->k_full[buf]);
          mbar_arrive_expect_tx(kf, C::kTileBytes);
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_3d(sbase + C::kKOff + buf * C::kTileBytes + sub * C::kSubBytes, &kmap, 64 * sub, j * kBN,
                        static_cast<int32_t>(head), kf);
        }
        const int slot = j % kScaleSlots;
        if (j >= kScaleSlots &&
            !wait_bounded<true>(smem_u32(&bars->sc_empty[slot]), ((j / kScaleSlots) & 1) ^ 1, err))
          break;
        scales[slot * kBN + tok_l] = j * kBN + tok_l < a.nk ? a.scale_log2 : 0.f;
        mbar_arrive(smem_u32(&bars->sc_full[slot]));
        if (tok_l == 0) {
          if (j >= kKvBufs && !wait_bounded<true>(smem_u32(&bars->v_empty[buf]), par, err)) break;
          const uint32_t vf = smem_u32(&bars->v_full[buf]);
          mbar_arrive_expect_tx(vf, C::kTileBytes);
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_3d(sbase + C::kVOff + buf * C::kTileBytes + sub * C::kSubBytes, &vmap, 64 * sub, j * kBN,
                        static_cast<int32_t>(head), vf);
        }
      }
    } else {
    // Cache row of token `tok` of this (sequence, kv-head): contiguous
    // [B, Hkv, capacity] or, through the page table, [pages, Hkv, 64];
    // -1 for a token in a missing page (flagged; its codes read as zero).
    const bool paged = cache.page_table != nullptr;
    const int64_t row0 = (static_cast<int64_t>(w.b) * cache.hkv + w.kvh) * cache.capacity;
    auto cache_row = [&](int tok) -> int64_t {
      if (!paged) return row0 + tok;
      const int page = __ldg(cache.page_table + static_cast<int64_t>(w.b) * cache.max_pages + tok / kPage);
      if (page < 0 || page >= cache.num_pages) return -1;
      return (static_cast<int64_t>(page) * cache.hkv + w.kvh) * kPage + tok % kPage;
    };
    const uint4 *kc = reinterpret_cast<const uint4 *>(cache.k_codes);
    const uint4 *vc = reinterpret_cast<const uint4 *>(cache.v_codes);
    const __half *ks = reinterpret_cast<const __half *>(cache.k_scales);
    const __half *vs = reinterpret_cast<const __half *>(cache.v_scales);
    // No prefetch across tiles: the two operand buffers let this warpgroup
    // run up to two tiles ahead of the tensor core, which hides the load.
    for (int j = 0; j < n; ++j) {
      const int tok = j * kBN + tok_l;
      uint4 ck[D / 32], cv[D / 32];
      float fk = 0.f;
      __half2 sv = __float2half2_rn(0.f);
      const int64_t row = tok < a.nk ? cache_row(tok) : -1;
      if (tok < a.nk && row < 0) atomicOr(err, kFlagBadPage);
      if (row >= 0) {
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          ck[i] = __ldg(kc + row * (D / 32) + i);
          cv[i] = __ldg(vc + row * (D / 32) + i);
        }
        fk = __half2float(ks[row]) * a.scale_log2;
        sv = __half2half2(vs[row]);
      } else {
#pragma unroll
        for (int i = 0; i < D / 32; ++i) ck[i] = cv[i] = make_uint4(0, 0, 0, 0);
      }
      const int buf = j % kKvBufs;
      const uint32_t par = ((j / kKvBufs) & 1) ^ 1;
      if (j >= kKvBufs && !wait_bounded<true>(smem_u32(&bars->k_empty[buf]), par, err)) break;
      store_row<D, false>(sbase + C::kKOff + buf * C::kTileBytes, tok_l, ck, sv);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars->k_full[buf]));
      const int slot = j % kScaleSlots;
      if (j >= kScaleSlots &&
          !wait_bounded<true>(smem_u32(&bars->sc_empty[slot]), ((j / kScaleSlots) & 1) ^ 1, err))
        break;
      scales[slot * kBN + tok_l] = fk;
      mbar_arrive(smem_u32(&bars->sc_full[slot]));
      if (j >= kKvBufs && !wait_bounded<true>(smem_u32(&bars->v_empty[buf]), par, err)) break;
      store_row<D, true>(sbase + C::kVOff + buf * C::kTileBytes, tok_l, cv, sv);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars->v_full[buf]));
    }
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
      if (!(ok = wait_bounded(smem_u32(&bars->sc_full[slot]), (j / kScaleSlots) & 1, err))) break;
      if (!(ok = wait_bounded(smem_u32(&bars->s_full[t]), j & 1, err))) break;
      tc_fence_after();
      const uint32_t kf = smem_u32(scales + slot * kBN);
      const int key0 = j * kBN;
      const bool masked = key0 + kBN - 1 > warp_limit;

      // The tile body is instantiated twice: with per-key masking (tiles
      // that cross the causal diagonal or the end of the keys) and without.
      float tsum = 0.f;
      auto tile = [&](auto mask_tag) {
        constexpr bool M = decltype(mask_tag)::value;
        if (j == 0) {  // the first tile fixes the reference maximum
          float mx = -INFINITY;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t s[32];
            tmem_ld32(s_tm + c * 32, s);
            mx = fmaxf(mx, chunk_max<M>(s, kf + c * 128, key0 + c * 32, limit));
          }
          m = mx == -INFINITY ? 0.f : mx;
        }
        // P chunk c (16 columns) overwrites S columns already read.
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t cur[32], h[16];
          tmem_ld32(s_tm + c * 32, cur);
          float cs = chunk_exp<M>(cur, kf + c * 128, m, key0 + c * 32, limit, h);
          if (__any_sync(0xffffffffu, !(cs <= static_cast<float>(kRedoSum)))) {
            // the reference maximum moves: rescale what was built on the old one
            const float mn = fmaxf(m, chunk_max<M>(cur, kf + c * 128, key0 + c * 32, limit));
            const float alpha = ex2(m - mn);
            m = mn, l *= alpha, tsum *= alpha;
            rescale_tmem<D>(s_tm, o_tm, c, j > 0, alpha);
            tmem_ld32(s_tm + c * 32, cur);  // S chunk c is intact: P so far only covers chunks < c/2
            cs = chunk_exp<M>(cur, kf + c * 128, m, key0 + c * 32, limit, h);
          }
          tsum += cs;
          tmem_st16(s_tm + c * 16, h);
        }
      };
      if (masked)
        tile(std::true_type{});
      else
        tile(std::false_type{});
      l += tsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full[t]));
      mbar_arrive(smem_u32(&bars->sc_empty[slot]));
    }

    // ------------------------------------------------------------ epilogue
    const bool done = wait_bounded(smem_u32(&bars->o_full), 0, err, ok ? kWaitCycles : kDrainCycles);
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
          // INT4: column 8q+p of O holds d = 8q + (0 4 1 5 2 6 3 7)[p]; KV16: d = 8q + p
          constexpr int e1 = KV16 ? 1 : 2, e2 = KV16 ? 2 : 4, e3 = KV16 ? 3 : 6, e4 = KV16 ? 4 : 1;
          constexpr int e5 = KV16 ? 5 : 3, e6 = KV16 ? 6 : 5, e7 = 7;
          const uint32_t h0 = pack_half2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + e1]) * inv);
          const uint32_t h1 = pack_half2(__uint_as_float(o[8 * q + e2]) * inv, __uint_as_float(o[8 * q + e3]) * inv);
          const uint32_t h2 = pack_half2(__uint_as_float(o[8 * q + e4]) * inv, __uint_as_float(o[8 * q + e5]) * inv);
          const uint32_t h3 = pack_half2(__uint_as_float(o[8 * q + e6]) * inv, __uint_as_float(o[8 * q + e7]) * inv);
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

template <int D, bool KV16>
cudaError_t launch_tc(const PrefillArgs &a, const KvView &cache, const CUtensorMap &qmap, const CUtensorMap &omap,
                      const CUtensorMap &kmap, const CUtensorMap &vmap, uint32_t *err, cudaStream_t stream) {
  using C = TcCfg<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, KV16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int G = a.hq / cache.hkv;
  const int nqb = (a.nq + kBM - 1) / kBM;
  const int64_t items = (G % 2 == 0) ? static_cast<int64_t>(a.batch) * cache.hkv * (G / 2) * nqb
                                     : static_cast<int64_t>(a.batch) * a.hq * ((nqb + 1) / 2);
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_tc_kernel<D, KV16><<<static_cast<unsigned>(items), kThreads, C::kSmem, stream>>>(a, cache, qmap, omap, kmap,
                                                                                           vmap, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, const KvView &cache, const CUtensorMap &qmap,
                           const CUtensorMap &omap, uint32_t *err, cudaStream_t stream) {
  if (a.batch == 0 || a.nq == 0) return cudaSuccess;
  return cache.head_dim == 128 ? launch_tc<128, false>(a, cache, qmap, omap, qmap, qmap, err, stream)
                               : launch_tc<64, false>(a, cache, qmap, omap, qmap, qmap, err, stream);
}

cudaError_t launch_prefill16(const PrefillArgs &a, int hkv, int head_dim, const CUtensorMap &qmap,
                             const CUtensorMap &omap, const CUtensorMap &kmap, const CUtensorMap &vmap, uint32_t *err,
                             cudaStream_t stream) {
  if (a.batch == 0 || a.nq == 0) return cudaSuccess;
  KvView cache = {};
  cache.hkv = hkv, cache.model_hkv = hkv, cache.head_dim = head_dim, cache.bits = 16;
  return head_dim == 128 ? launch_tc<128, true>(a, cache, qmap, omap, kmap, vmap, err, stream)
                         : launch_tc<64, true>(a, cache, qmap, omap, kmap, vmap, err, stream);
}

}  // namespace qattn
