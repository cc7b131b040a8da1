// pq.cu -- progressive INT8 -> INT4 KV storage and the decode over it.
//
// TurboAttention (arXiv 2412.08585) §3.1 (Blockwise Progressive Quantization):
// each 64-token sub-block of K or V is first quantized to 8 bits
// symmetrically with one FP16 scale, then stored channel-wise as asymmetric
// 4-bit codes whose integer scale and zero point are kept in INT8; reading a
// block back is INT4 -> INT8 (q2 * s2 + z2) and then the FP16 scale.  The
// page's equations are missing; the reading taken (every step exact):
//   s1 = fp16(fp32(absmax(block) / 127)), q1 = clamp(RNE(x / s1), -127, 127)
//   per channel: lo = min q1, hi = max q1, s2 = max(1, ceil((hi - lo) / 15)),
//   z2 = lo, q2 = RNE((q1 - lo) / s2) in [0, 15]
//
// pq_quantize_kernel   one CTA of D threads (one per channel) per 64-token
//                      block of one (sequence, kv-head) and tensor: stage 1
//                      (block absmax, int8 codes), stage 2 (each thread's
//                      channel), nibble packing by shuffles
// decode_pq_kernel     split-KV decode, one CTA per (key range, sequence,
//                      kv-head): a producer thread streams whole blocks
//                      (four per stage: codes + parameter records) by bulk
//                      copies into a 2-deep ring; each of 16 consumer warps
//                      (4 per block) rebuilds its 16 tokens' exact
//                      integer values q1' in fp16 in a private swizzled tile
//                      (the block's stage is released right after), then
//                      S^T = q1'_K . Q^T by mma.sync (tokens on M), S scaled
//                      by the block's s1_K, an online softmax, and
//                      O^T += q1'_V^T . (P s1_V)^T; warps merge in shared
//                      memory laid over the ring, ranges by the combine
//                      kernel.  The work is latency-bound: 16 warps an SM
//                      measured faster than 12 and those than 8.
#include <math.h>

#include "../../include/qattn.h"
#include "internal.h"
#include "ptx.cuh"
#include "quant_row.cuh"

namespace qattn {
namespace {

constexpr int kPqBlock = 64;  // tokens per block

__device__ __forceinline__ __half lds_half(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __ushort_as_half(v);
}

// ------------------------------------------------------------------ quantize
template <typename T, int D>
__global__ void __launch_bounds__(D)
    pq_quantize_kernel(const T *__restrict__ k, const T *__restrict__ v, int n, const int32_t *__restrict__ start_block,
                       PqView c, uint32_t *err) {
  __shared__ float red[D / 32];
  const int blk = blockIdx.x, bh = blockIdx.y;
  const bool is_v = blockIdx.z != 0;
  const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const int b = bh / c.hkv;
  const int64_t dst_blk = static_cast<int64_t>(start_block ? __ldg(start_block + b) : 0) + blk;
  if (dst_blk < 0 || dst_blk >= c.capacity / kPqBlock) {  // block-uniform
    if (d == 0) atomicOr(err, kFlagBadPage);
    return;
  }
  const T *src = (is_v ? v : k) + (static_cast<int64_t>(bh) * n + static_cast<int64_t>(blk) * kPqBlock) * D + d;
  float x[kPqBlock];
  float am = 0.f;
#pragma unroll
  for (int t = 0; t < kPqBlock; ++t) {
    x[t] = static_cast<float>(src[static_cast<int64_t>(t) * D]);
    am = fmaxf(am, fabsf(x[t]));
  }
  // stage 1: the block's absmax -> s1, int8 codes
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  if (lane == 0) red[warp] = am;
  __syncthreads();
  am = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) am = fmaxf(am, red[w]);
  const __half s1 = universal_scale(am);
  const float u = __half2float(s1);
  // stage 2: this thread's channel
  int lo = 127, hi = -127;
#pragma unroll
  for (int t = 0; t < kPqBlock; ++t) {
    const int q1 = code8(x[t], u);
    lo = min(lo, q1), hi = max(hi, q1);
  }
  const int s2 = max(1, (hi - lo + 14) / 15);
  const int64_t row0 = (static_cast<int64_t>(bh) * c.capacity) + dst_blk * kPqBlock;
  uint8_t *codes = (is_v ? c.v_codes : c.k_codes) + row0 * (D / 2) + d / 2;
#pragma unroll
  for (int t = 0; t < kPqBlock; ++t) {
    const int num = code8(x[t], u) - lo;  // 0 .. hi - lo
    const int fl = num / s2, rem = num - fl * s2;
    const int q2 = fl + ((2 * rem > s2) || (2 * rem == s2 && (fl & 1)) ? 1 : 0);
    const int partner = __shfl_xor_sync(0xffffffffu, q2, 1);
    if ((d & 1) == 0) codes[static_cast<int64_t>(t) * (D / 2)] = static_cast<uint8_t>(q2 | (partner << 4));
  }
  uint8_t *rec = (is_v ? c.v_params : c.k_params) + (static_cast<int64_t>(bh) * (c.capacity / kPqBlock) + dst_blk) * (2 * D + 16);
  rec[d] = static_cast<uint8_t>(s2);
  rec[D + d] = static_cast<uint8_t>(static_cast<int8_t>(lo));
  if (d < 8) reinterpret_cast<uint16_t *>(rec + 2 * D)[d] = d == 0 ? __half_as_ushort(s1) : 0;
}

// ------------------------------------------- a full decode buffer -> block
// One CTA of D threads (one per channel) per sequence whose buffer holds 64
// rows: each (kv-head, tensor)'s int8 codes are stage 1 already (universal
// scale u = s1), so only stage 2 runs; the block goes to position
// cache_lens[b] (a multiple of 64); then the buffer empties.  R and u are
// left as they are: the universal range already bounds the block.
template <int D>
__global__ void __launch_bounds__(D) flashq_flush_pq_kernel(FlashqView f, PqView c, const int32_t *__restrict__ cache_lens,
                                                           uint32_t *err) {
  const int b = blockIdx.x, d = threadIdx.x;
  if (f.count[b] < kPqBlock) return;  // uniform across the block
  const int64_t pos = __ldg(cache_lens + b);
  const bool fits = pos >= 0 && pos % kPqBlock == 0 && pos + kPqBlock <= c.capacity;
  if (!fits && d == 0) atomicOr(err, kFlagBadPage);
  const int64_t blk = pos / kPqBlock;
  for (int it = 0; fits && it < 2 * f.hkv; ++it) {
    const int h = it >> 1, t = it & 1;
    const int64_t bh = static_cast<int64_t>(b) * f.hkv + h;
    const int8_t *src = (t ? f.v_codes : f.k_codes) + bh * kPqBlock * D + d;
    int q1[kPqBlock];
    int lo = 127, hi = -127;
#pragma unroll
    for (int r = 0; r < kPqBlock; ++r) {
      q1[r] = src[r * D];
      lo = min(lo, q1[r]), hi = max(hi, q1[r]);
    }
    const int s2 = max(1, (hi - lo + 14) / 15);
    uint8_t *codes = (t ? c.v_codes : c.k_codes) + (bh * c.capacity + blk * kPqBlock) * (D / 2) + d / 2;
#pragma unroll
    for (int r = 0; r < kPqBlock; ++r) {
      const int num = q1[r] - lo;
      const int fl = num / s2, rem = num - fl * s2;
      const int q2 = fl + ((2 * rem > s2) || (2 * rem == s2 && (fl & 1)) ? 1 : 0);
      const int partner = __shfl_xor_sync(0xffffffffu, q2, 1);
      if ((d & 1) == 0) codes[static_cast<int64_t>(r) * (D / 2)] = static_cast<uint8_t>(q2 | (partner << 4));
    }
    uint8_t *rec = (t ? c.v_params : c.k_params) + (bh * (c.capacity / kPqBlock) + blk) * (2 * D + 16);
    rec[d] = static_cast<uint8_t>(s2);
    rec[D + d] = static_cast<uint8_t>(static_cast<int8_t>(lo));
    if (d < 8) reinterpret_cast<uint16_t *>(rec + 2 * D)[d] = d == 0 ? (t ? f.v_scale : f.k_scale)[bh] : 0;
  }
  __syncthreads();  // every thread has read the buffer
  if (d == 0) f.count[b] = 0;
}

// -------------------------------------------------------------------- decode
constexpr int kWq = 16;                 // consumer warps, 16 tokens each: 4 per block, 4 blocks a stage
constexpr int kBlocksPerStage = 4;
constexpr int kThreadsPq = (kWq + 1) * 32;

template <int D>
struct Cq {
  static constexpr int kCodeBytes = kPqBlock * D / 2;       // one tensor's codes of a block
  static constexpr int kRec = 2 * D + 16;                   // one tensor's parameter record
  // stage: K codes, V codes (4 blocks each), K records, V records (4 each)
  static constexpr int kKOff = 0, kVOff = kBlocksPerStage * kCodeBytes;
  static constexpr int kKpOff = 2 * kBlocksPerStage * kCodeBytes, kVpOff = kKpOff + kBlocksPerStage * kRec;
  static constexpr int kStageBytes = (kVpOff + kBlocksPerStage * kRec + 127) / 128 * 128;
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr int kTileBytes = 16 * D * 2;             // 16 tokens x D fp16
  static constexpr int kPitch = D + 4;
  // the warps' merge area is laid over the ring once every stage is read
  static constexpr int kMergeBytes = kWq * 8 * kPitch * 4;
  static_assert(kMergeBytes <= kStages * kStageBytes, "the merge area fits the ring");
  static constexpr int kSmem = kStages * kStageBytes + kWq * 2 * kTileBytes + 2 * kWq * 8 * 4 +
                               2 * kStages * 8 + 16 + 1024;
  // the rebuild: a lane keeps 8 channels of kTokLane tokens, the warp's
  // kGroups lane groups taking interleaved tokens (the groups' code rows then
  // sit D/2 bytes apart: distinct banks)
  static constexpr int kLanesRow = D / 8, kGroups = 32 / kLanesRow, kTokLane = 16 / kGroups;
};

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// A warp tile: 16 token rows of D fp16, in 64-column subtiles of 16 x 128
// bytes whose 16-byte chunks are XOR-swizzled by the row (conflict-free
// ldmatrix).
template <int D>
__device__ __forceinline__ uint32_t wtile_addr(uint32_t tile, int tok, int chunk) {
  return tile + (chunk >> 3) * (16 * 128) + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
}

// The s2 and z2 of eight channels as four fp16 pairs each (exact small
// integers: bytes become the fp16 integers 1024 + v by bit placement; z2 is
// biased by 128 so that every byte is unsigned).
struct Params8 {
  __half2 s[4], z[4];
};
__device__ __forceinline__ Params8 params8(uint2 s2, uint2 z2) {
  Params8 p;
  const uint32_t sb[2] = {s2.x, s2.y}, zb[2] = {z2.x ^ 0x80808080u, z2.y ^ 0x80808080u};
  const __half2 k1024 = __float2half2_rn(1024.f), k1152 = __float2half2_rn(1152.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = 2 * (k & 1);  // byte of the word holding channel 2k
    const uint32_t sp = lop3_and_xor(__byte_perm(sb[k >> 1], 0, e | ((e + 1) << 8)), 0x00FF00FFu, 0x64006400u);
    const uint32_t zp = lop3_and_xor(__byte_perm(zb[k >> 1], 0, e | ((e + 1) << 8)), 0x00FF00FFu, 0x64006400u);
    p.s[k] = __hsub2(*reinterpret_cast<const __half2 *>(&sp), k1024);
    p.z[k] = __hsub2(*reinterpret_cast<const __half2 *>(&zp), k1152);
  }
  return p;
}

// Eight channels of one token: code word w (eight unsigned nibbles, element
// 2k in the low nibble of byte k) -> q1' = q2 * s2 + z2 as four fp16 pairs in
// element order, exactly.
__device__ __forceinline__ uint4 rebuild8(uint32_t w, const Params8 &p) {
  const uint32_t w4 = w >> 4;
  const __half2 k1024 = __float2half2_rn(1024.f);
  uint32_t r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // (element 2k, 2k + 1): byte k's low nibble, byte k's high nibble
    const uint32_t qp = lop3_and_xor(__byte_perm(w, w4, k | ((k + 4) << 8)), 0x000F000Fu, 0x64006400u);
    const __half2 y = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&qp), k1024), p.s[k], p.z[k]);
    r[k] = *reinterpret_cast<const uint32_t *>(&y);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

template <int D>
__global__ void __launch_bounds__(kThreadsPq, 1)
    decode_pq_kernel(const uint16_t *__restrict__ q, const int32_t *__restrict__ seq_lens, int batch, int hq, PqView c,
                     int chunk, float scale_log2, uint16_t *__restrict__ out, float *__restrict__ lse,
                     float *__restrict__ partial_o, float *__restrict__ partial_lse, uint32_t *err) {
  using C = Cq<D>;
  constexpr int kMt = D / 16;
  constexpr int kStageTok = kBlocksPerStage * kPqBlock;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *tiles = smem + C::kStages * C::kStageBytes;                     // [warp][K, V] tiles
  float *mo = reinterpret_cast<float *>(smem);  // [warp][head][kPitch], over the ring after the last stage
  float *mm = reinterpret_cast<float *>(tiles + kWq * 2 * C::kTileBytes);
  float *ml = mm + kWq * 8;
  uint64_t *full = reinterpret_cast<uint64_t *>(ml + kWq * 8);
  uint64_t *empty = full + C::kStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, splits = gridDim.x;
  const int bh = blockIdx.y, b = bh / c.hkv, kvh = bh % c.hkv;
  const int G = hq / c.hkv;
  const int64_t len = min(static_cast<int64_t>(max(__ldg(seq_lens + b), 0)), c.capacity);
  const int64_t t0 = static_cast<int64_t>(split) * chunk;
  const int64_t t1 = min(t0 + chunk, len);
  const int nblk = t1 > t0 ? static_cast<int>((t1 - t0 + kPqBlock - 1) / kPqBlock) : 0;  // blocks of the range
  const int nst = (nblk + kBlocksPerStage - 1) / kBlocksPerStage;
  const int64_t row0 = static_cast<int64_t>(b) * hq + static_cast<int64_t>(kvh) * G;  // first q-head row

  if (nst == 0) {  // no key in this range: an empty partial (or, unsplit, O = 0)
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
      mbar_init(smem_u32(empty + s), kWq);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kWq) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int64_t blk0 = t0 / kPqBlock;
      const int64_t nblk_cap = c.capacity / kPqBlock;
      for (int j = 0; j < nst; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages &&
            !mbar_wait(smem_u32(empty + s), ((j / C::kStages) & 1) ^ 1, err, *abort_flag ? kDrainCycles : kWaitCycles)) {
          *abort_flag = 1;
          break;
        }
        // the stage's blocks are consecutive: one copy per tensor for the codes, one for the records
        const int nb = min(kBlocksPerStage, nblk - j * kBlocksPerStage);
        const uint32_t st = smem_u32(smem + s * C::kStageBytes), bar = smem_u32(full + s);
        const int64_t blk = blk0 + static_cast<int64_t>(j) * kBlocksPerStage;
        const int64_t crow = static_cast<int64_t>(bh) * c.capacity + blk * kPqBlock;
        const int64_t prec = static_cast<int64_t>(bh) * nblk_cap + blk;
        mbar_arrive_expect_tx(bar, nb * (2 * C::kCodeBytes + 2 * C::kRec));
        bulk_g2s(st + C::kKOff, c.k_codes + crow * (D / 2), nb * C::kCodeBytes, bar);
        bulk_g2s(st + C::kVOff, c.v_codes + crow * (D / 2), nb * C::kCodeBytes, bar);
        bulk_g2s(st + C::kKpOff, c.k_params + prec * C::kRec, nb * C::kRec, bar);
        bulk_g2s(st + C::kVpOff, c.v_params + prec * C::kRec, nb * C::kRec, bar);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // warp w: block w / 4 of each stage, its tokens 16 (w % 4) .. + 15
  const int wb = warp >> 2, wt = (warp & 3) * 16;
  const int g = lane >> 2, cc = lane & 3;
  uint32_t qb[kMt][2];  // Q^T as the B operand: k-step kk covers d = 16 kk ..; column g is q-head g
  {
    const uint32_t *qr = reinterpret_cast<const uint32_t *>(q + (row0 + min(g, G - 1)) * D);
#pragma unroll
    for (int kk = 0; kk < kMt; ++kk) {
      qb[kk][0] = g < G ? __ldg(qr + 8 * kk + cc) : 0u;
      qb[kk][1] = g < G ? __ldg(qr + 8 * kk + 4 + cc) : 0u;
    }
  }
  float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f;
  float o[kMt][4];
#pragma unroll
  for (int mt = 0; mt < kMt; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  const uint32_t ktile = smem_u32(tiles + warp * 2 * C::kTileBytes), vtile = ktile + C::kTileBytes;
  // the rebuild: lane keeps channels 8 (lane % kLanesRow) .. + 7 of tokens
  // rgrp, rgrp + kGroups, ... of the warp's 16 (rgrp = lane / kLanesRow)
  const int rch = 8 * (lane % C::kLanesRow), rgrp = lane / C::kLanesRow;
  const int mq = lane >> 3;
  const int ktok = (lane & 7) + (mq & 1) * 8, kch = mq >> 1;   // ldmatrix rows of K (non-transposed)
  const int vtok = (lane & 7) + (mq >> 1) * 8, vch = mq & 1;   // and of V (transposed)

  for (int j = 0; j < nst; ++j) {
    const int s = j % C::kStages;
    const bool got = mbar_wait(smem_u32(full + s), (j / C::kStages) & 1, err, *abort_flag ? kDrainCycles : kWaitCycles);
    if (!got) *abort_flag = 1;
    const int64_t tok0 = t0 + static_cast<int64_t>(j) * kStageTok + wb * kPqBlock + wt;
    const int nvalid = got ? static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(16), t1 - tok0))) : 0;
    float s1k = 0.f, s1v = 0.f;
    if (nvalid > 0) {
      // rebuild q1' of this warp's 16 tokens into its tiles, then release the stage
      const uint32_t st = smem_u32(smem + s * C::kStageBytes);
      const uint32_t kp = st + C::kKpOff + wb * C::kRec, vp = st + C::kVpOff + wb * C::kRec;
      s1k = __half2float(lds_half(kp + 2 * D)) * scale_log2;
      s1v = __half2float(lds_half(vp + 2 * D)) * 0.00390625f;  // carries 2^-8: p * s1_V stays in fp16 range
      __syncwarp();  // every lane has finished reading the tiles of the previous block
#pragma unroll
      for (int t = 0; t < 2; ++t) {  // K, V
        const uint32_t pr = t ? vp : kp;
        const Params8 p8 = params8(lds64(pr + rch), lds64(pr + D + rch));
        const uint32_t codes = st + (t ? C::kVOff : C::kKOff) + wb * C::kCodeBytes + (wt + rgrp) * (D / 2) + rch / 2;
        const uint32_t tile = t ? vtile : ktile;
#pragma unroll
        for (int i = 0; i < C::kTokLane; ++i) {
          uint32_t w;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(codes + i * C::kGroups * (D / 2)));
          const uint4 y = rebuild8(w, p8);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(wtile_addr<D>(tile, rgrp + i * C::kGroups, rch >> 3)),
                       "r"(y.x), "r"(y.y), "r"(y.z), "r"(y.w)
                       : "memory");
        }
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(smem_u32(empty + s));  // the stage is no longer read by this warp
    if (nvalid > 0) {
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < kMt; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm4(wtile_addr<D>(ktile, ktok, 2 * kk + kch), a0, a1, a2, a3);
        if (kk & 1)
          mma_16816(sb, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        else
          mma_16816(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
      // scores (log2 units) of tokens g, g + 8 for q-heads 2cc, 2cc + 1
      float ts0 = (sa[0] + sb[0]) * s1k, ts1 = (sa[1] + sb[1]) * s1k;
      float ts2 = (sa[2] + sb[2]) * s1k, ts3 = (sa[3] + sb[3]) * s1k;
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
      l0 += p0 + p2, l1 += p1 + p3;
      const uint32_t r0 = pack_half2(p0 * s1v, p1 * s1v), r1 = pack_half2(p2 * s1v, p3 * s1v);
      const uint32_t pb0 = movmatrix_trans(r0), pb1 = movmatrix_trans(r1);
      // tokens past the keys: their rebuilt V values are finite, their P is 0
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(wtile_addr<D>(vtile, vtok, 2 * mt + vch), a0, a1, a2, a3);
        mma_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
      }
    }
  }

  // ----------------------------------------------------- merge the warps
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWq * 32) : "memory");  // every warp is done with the ring
  float *mw = mo + warp * 8 * C::kPitch;
#pragma unroll
  for (int mt = 0; mt < kMt; ++mt) {  // O^T carried s1_V * 2^-8: the 2^8 returns here
    mw[(2 * cc) * C::kPitch + 16 * mt + g] = o[mt][0] * 256.f;
    mw[(2 * cc + 1) * C::kPitch + 16 * mt + g] = o[mt][1] * 256.f;
    mw[(2 * cc) * C::kPitch + 16 * mt + g + 8] = o[mt][2] * 256.f;
    mw[(2 * cc + 1) * C::kPitch + 16 * mt + g + 8] = o[mt][3] * 256.f;
  }
  if (g == 0) {
    mm[warp * 8 + 2 * cc] = m0, mm[warp * 8 + 2 * cc + 1] = m1;
    ml[warp * 8 + 2 * cc] = l0, ml[warp * 8 + 2 * cc + 1] = l1;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWq * 32) : "memory");
  for (int i = threadIdx.x; i < G * D; i += kWq * 32) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWq; ++w)
      if (ml[w * 8 + h] > 0.f) M = fmaxf(M, mm[w * 8 + h]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWq; ++w) {
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

template <typename T, int D>
cudaError_t launch_pq_quantize_t(const void *k, const void *v, int batch, int n, const int32_t *start_block,
                                 const PqView &c, uint32_t *err, cudaStream_t stream) {
  dim3 grid(n / kPqBlock, batch * c.hkv, 2);
  pq_quantize_kernel<T, D><<<grid, D, 0, stream>>>(static_cast<const T *>(k), static_cast<const T *>(v), n,
                                                     start_block, c, err);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_pq_t(const DecodePqArgs &a, const PqView &c, uint32_t *err, cudaStream_t stream) {
  using C = Cq<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_pq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(a.splits, a.batch * c.hkv);
  float *po = a.splits > 1 ? a.partial_o : nullptr;
  float *pl = a.splits > 1 ? a.partial_lse : nullptr;
  decode_pq_kernel<D><<<grid, kThreadsPq, C::kSmem, stream>>>(a.q, a.seq_lens, a.batch, a.hq, c, a.chunk,
                                                              a.scale_log2, a.out, a.lse, po, pl, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  return launch_combine(a.partial_o, a.partial_lse, a.splits, static_cast<int64_t>(a.batch) * a.hq, D, a.out, a.lse,
                        false, stream);
}

}  // namespace

cudaError_t launch_pq_quantize(const void *k, const void *v, bool fp16_in, int batch, int n, const int32_t *start_block,
                               const PqView &c, uint32_t *err, cudaStream_t stream) {
  if (batch == 0 || n == 0) return cudaSuccess;
  if (c.head_dim == 128)
    return fp16_in ? launch_pq_quantize_t<__half, 128>(k, v, batch, n, start_block, c, err, stream)
                   : launch_pq_quantize_t<float, 128>(k, v, batch, n, start_block, c, err, stream);
  return fp16_in ? launch_pq_quantize_t<__half, 64>(k, v, batch, n, start_block, c, err, stream)
                 : launch_pq_quantize_t<float, 64>(k, v, batch, n, start_block, c, err, stream);
}

cudaError_t launch_flashq_flush_pq(const FlashqView &f, const PqView &c, const int32_t *cache_lens, int batch,
                                   uint32_t *err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  if (c.head_dim == 128)
    flashq_flush_pq_kernel<128><<<batch, 128, 0, stream>>>(f, c, cache_lens, err);
  else
    flashq_flush_pq_kernel<64><<<batch, 64, 0, stream>>>(f, c, cache_lens, err);
  return cudaGetLastError();
}

cudaError_t launch_decode_pq(const DecodePqArgs &a, const PqView &c, uint32_t *err, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  return c.head_dim == 128 ? launch_decode_pq_t<128>(a, c, err, stream) : launch_decode_pq_t<64>(a, c, err, stream);
}

}  // namespace qattn
