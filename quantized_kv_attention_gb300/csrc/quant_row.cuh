// quant_row.cuh -- quantization of one K or V row (D values) by one warp,
// shared by the append kernel and the fused append + decode step so that
// both write the same bits.
//
// TurboAttention (arXiv 2412.08585) §2.3: symmetric quantization, zero point
// 0; "Quantized Cross-Attention ... In-SRAM Dequantization" §3.2: 4-bit codes
// with one FP16 scale per token.  s = fp16(fp32(absmax / 7)), both roundings
// to nearest even, saturating at 65504; code = round-half-even(x / s) clamped
// to [-7, 7] on the exact quotient: a candidate from one fused multiply-add,
// proved by its exact remainder, and for the values it cannot prove (ties)
// exact comparisons with the half-way points (k + 1/2) s, which are exact in
// fp32 (s has 11 significant bits, 2k + 1 at most 4 bits).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace qattn {

template <typename T, int VPL>
struct RowLoad;

template <>
struct RowLoad<float, 4> {
  static __device__ __forceinline__ void load(const float *p, float (&x)[4]) {
    float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  }
};
template <>
struct RowLoad<float, 2> {
  static __device__ __forceinline__ void load(const float *p, float (&x)[2]) {
    float2 v = __ldg(reinterpret_cast<const float2 *>(p));
    x[0] = v.x, x[1] = v.y;
  }
};
template <>
struct RowLoad<__half, 4> {
  static __device__ __forceinline__ void load(const __half *p, float (&x)[4]) {
    uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
    float2 a = __half22float2(*reinterpret_cast<__half2 *>(&v.x));
    float2 b = __half22float2(*reinterpret_cast<__half2 *>(&v.y));
    x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
  }
};
template <>
struct RowLoad<__half, 2> {
  static __device__ __forceinline__ void load(const __half *p, float (&x)[2]) {
    uint32_t v = __ldg(reinterpret_cast<const unsigned int *>(p));
    float2 a = __half22float2(*reinterpret_cast<__half2 *>(&v));
    x[0] = a.x, x[1] = a.y;
  }
};

// Round-half-even of |x| / s on the exact quotient, clamped to 7: count the
// half-way points (2j+1) s / 2 below |x|; at an exact half-way point round to
// the even neighbour, i.e. count that point only when j is odd.
__device__ __forceinline__ int code_of(float x, float s) {
  const float ax = fabsf(x);
  const float h = 0.5f * s;
  int m = (ax > h) + (ax >= 3.f * h) + (ax > 5.f * h) + (ax >= 7.f * h) + (ax > 9.f * h) +
          (ax >= 11.f * h) + (ax > 13.f * h);
  return x < 0.f ? -m : m;
}

// min / max that return NaN when either operand is NaN.
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The lane's VPL codes clamp(RNE(x / s), -7, 7) as packed nibbles (element j
// at bits 4j), for s > 0 -- the same codes as code_of, with fewer
// instructions.  A fused multiply-add of x with r ~ 1/s and 1.5 * 2^23
// rounds x * r to an integer m (the sum has ulp 1), and the sum's encoding is
// 0x4B400000 + m, whose low nibble is m in two's complement.  Because r is an
// approximation, m is then proved: with e = x - m s taken by a second fused
// multiply-add, |e| < s / 2 means m is the integer nearest to x / s (a
// computed |e| below the representable s / 2 implies the exact one is, as
// rounding is monotonic).  A value at or past a half-way point -- an exact tie
// or a candidate off by one -- and a NaN (it fails the test) are coded by the
// threshold count instead.  kClamp first clamps x to [-7s, 7s], which leaves
// the clamped code unchanged; it is needed only when s may be far below
// absmax / 7: a subnormal or saturated fp16 scale.  For a normal scale below
// 65504, s >= (absmax / 7)(1 - 2^-24)(1 - 2^-11), so |x| / s <= 7.004 and m
// stays in [-7, 7] without it.
template <int VPL, bool kClamp>
__device__ __forceinline__ uint32_t codes4(const float (&x)[VPL], float s) {
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  const float lim = 7.f * s, h = 0.5f * s;
  // The nibbles are summed as integers: sum_j enc(y_j) 16^j = 0x4B400000 *
  // ones + sum_j m_j 16^j (ones = sum_j 16^j, modulo 2^32); adding
  // (8 - 0x4B400000) * ones leaves sum_j (m_j + 8) 16^j with every digit in
  // [1, 15] (no carries), and m_j + 8 XOR 8 is m_j's two's-complement nibble.
  static_assert(VPL == 2 || VPL == 4, "two or four values per lane");
  constexpr uint32_t kOnes = VPL == 4 ? 0x1111u : 0x11u;
  constexpr uint32_t kBias = (8u - 0x4B400000u) * kOnes;
  uint32_t acc = kBias;
  bool sure = true;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const float xc = kClamp ? fmax_nan(fmin_nan(x[j], lim), -lim) : x[j];
    const float y = fmaf(xc, r, kShift);
    const float e = fmaf(kShift - y, s, xc);
    sure = sure && fabsf(e) < h;
    acc += __float_as_uint(y) * (1u << (4 * j));
  }
  uint32_t packed = (acc ^ (8u * kOnes)) & (kOnes * 0xFu);
  if (!sure) {
    packed = 0;
#pragma unroll
    for (int j = 0; j < VPL; ++j) packed |= static_cast<uint32_t>(code_of(x[j], s) & 0xF) << (4 * j);
  }
  return packed;
}

// codes4 for any scale s >= 0 (all codes 0 when s == 0): the clamp only for
// a subnormal or saturated s.
template <int VPL>
__device__ __forceinline__ uint32_t codes4_any(const float (&x)[VPL], float s) {
  if (s >= 6.103515625e-05f && s < 65504.f) return codes4<VPL, false>(x, s);  // normal fp16 (2^-14 ..)
  return s > 0.f ? codes4<VPL, true>(x, s) : 0u;
}

// Quantizes one row of D values held by the 32 lanes of a warp: lane i
// holds elements 4i..4i+3 (D = 128) or 2i, 2i+1 (D = 64) in x and writes
// their packed nibbles (low nibble = even element) to dst_codes + i * D / 64;
// lane 0 writes the fp16 scale, which every lane gets back.  Every lane of
// the warp must call it.
template <int D>
__device__ __forceinline__ __half quantize_vals_warp(const float (&x)[D / 32], uint8_t *dst_codes,
                                                     uint16_t *dst_scale, int lane) {
  constexpr int VPL = D / 32;  // values per lane
  float am = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) am = fmaxf(am, fabsf(x[j]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));

  __half hs = __float2half_rn(__fdiv_rn(am, 7.0f));
  if (__hisinf(hs)) hs = __ushort_as_half(0x7BFF);
  const float s = __half2float(hs);

  const uint32_t packed = codes4_any<VPL>(x, s);
  uint8_t *dst = dst_codes + lane * (VPL / 2);
  if constexpr (VPL == 4)
    *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
  else
    *dst = static_cast<uint8_t>(packed);
  if (lane == 0) *dst_scale = __half_as_ushort(hs);
  return hs;
}

// Packed fp32 pairs: two IEEE round-to-nearest operations per instruction,
// no flush to zero, so the same bits as the scalar forms.
__device__ __forceinline__ uint64_t pair_of(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void pair_split(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t pair_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pair_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Four rows at once, one per group of 8 lanes (g = lane / 8, l = lane % 8),
// with the codes of quantize_vals_warp (the same bits): the row's D values
// are C = D / 32 chunks of 32, and lane l holds values 4l .. 4l + 3 of each
// chunk, x[c] being the group's chunk (c + g) % C (the rotation keeps the
// groups' shared-memory reads of a 16-lane phase on distinct banks).  The
// absmax takes three shuffle levels inside the group, the scale one division
// per lane for four rows.  For a normal fp16 scale the one-FMA coding of
// codes4 runs on pairs of values (y = x * rcp(s) + 1.5 * 2^23, m = y - 1.5 *
// 2^23, e = x - m * s, all exact but y), and the lane's values are exact when
// the largest |e| is below s / 2 (a NaN remainder fails the test); otherwise,
// and for other scales, codes4_any codes the chunks.  Lane l stores the
// nibbles of its values of chunk cc at byte 16 cc + 2l of the row, lane 0 of
// the group the scale.  A group whose dst_codes is null stores nothing.
// Every lane of the warp must call it.
template <int D>
__device__ __forceinline__ void quantize_vals_warp4(const float (&x)[D / 32][4], uint8_t *dst_codes,
                                                    uint16_t *dst_scale, int lane) {
  constexpr int C = D / 32;
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
  constexpr uint32_t kBias = (8u - 0x4B400000u) * 0x1111u;  // see codes4
  const int g = lane >> 3, l = lane & 7;
  float am = 0.f;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    am = fmaxf(am, fmaxf(fabsf(x[c][0]), fabsf(x[c][1])));
    am = fmaxf(am, fmaxf(fabsf(x[c][2]), fabsf(x[c][3])));
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  __half hs = __float2half_rn(__fdiv_rn(am, 7.0f));
  if (__hisinf(hs)) hs = __ushort_as_half(0x7BFF);
  const float s = __half2float(hs);
  if (dst_codes == nullptr) return;
  uint32_t packed[C];
  bool exact = false;
  if (s >= 6.103515625e-05f && s < 65504.f) {  // normal fp16 scale: |x| / s <= 7.004, no clamp
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
    const uint64_t r2 = pair_of(r, r), shift2 = pair_of(kShift, kShift), unshift2 = pair_of(-kShift, -kShift);
    const uint64_t ns2 = pair_of(-s, -s);
    float emax = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const uint64_t x01 = pair_of(x[c][0], x[c][1]), x23 = pair_of(x[c][2], x[c][3]);
      const uint64_t y01 = pair_fma(x01, r2, shift2), y23 = pair_fma(x23, r2, shift2);
      const uint64_t e01 = pair_fma(pair_add(y01, unshift2), ns2, x01);
      const uint64_t e23 = pair_fma(pair_add(y23, unshift2), ns2, x23);
      float e0, e1, e2, e3, y0, y1, y2, y3;
      pair_split(e01, e0, e1), pair_split(e23, e2, e3), pair_split(y01, y0, y1), pair_split(y23, y2, y3);
      emax = fmax_nan(fmax_nan(emax, fabsf(e0)), fmax_nan(fabsf(e1), fmax_nan(fabsf(e2), fabsf(e3))));
      const uint32_t acc = kBias + __float_as_uint(y0) + (__float_as_uint(y1) << 4) + (__float_as_uint(y2) << 8) +
                           (__float_as_uint(y3) << 12);
      packed[c] = (acc ^ 0x8888u) & 0xFFFFu;
    }
    exact = emax < 0.5f * s;
  }
  if (!exact) {
#pragma unroll
    for (int c = 0; c < C; ++c) packed[c] = codes4_any<4>(x[c], s);
  }
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int cc = (c + g) & (C - 1);
    *reinterpret_cast<uint16_t *>(dst_codes + cc * 16 + 2 * l) = static_cast<uint16_t>(packed[c]);
  }
  if (l == 0) *dst_scale = __half_as_ushort(hs);
}

// quantize_vals_warp of row `src` (D values of type T, lane i reading its
// elements as above).
template <typename T, int D>
__device__ __forceinline__ void quantize_row_warp(const T *src, uint8_t *dst_codes, uint16_t *dst_scale,
                                                  int lane) {
  float x[D / 32];
  RowLoad<T, D / 32>::load(src + lane * (D / 32), x);
  quantize_vals_warp<D>(x, dst_codes, dst_scale, lane);
}

// The int8 code of TurboAttention's 8-bit symmetric stage (§3.2, §3.3), shared
// by the decode buffer and the progressive blocks: a range R gives the scale
// u = fp16(fp32(R / 127)), saturating at 65504, and a value x the code
// clamp(RNE(x / u), -127, 127) on the exact quotient: the fp32 quotient gives
// a candidate m for |x| / u, corrected against the half-way points
// (m +- 1/2) u, which are exact in fp32 (at most 9 + 11 significant bits).
__device__ __forceinline__ __half universal_scale(float r) {
  __half u = __float2half_rn(__fdiv_rn(r, 127.0f));
  if (__hisinf(u)) u = __ushort_as_half(0x7BFF);
  return u;
}

__device__ __forceinline__ int code8(float x, float u) {
  if (!(u > 0.f)) return 0;
  const float ax = fabsf(x);
  float m = rintf(__fdiv_rn(ax, u));
  if (m >= 128.f) return x < 0.f ? -127 : 127;
  const float hi = (m + 0.5f) * u, lo = (m - 0.5f) * u;
  const bool odd = (static_cast<int>(m) & 1) != 0;
  if (ax > hi || (ax == hi && odd)) m += 1.f;
  else if (m >= 1.f && (ax < lo || (ax == lo && odd))) m -= 1.f;
  const int c = min(static_cast<int>(m), 127);
  return x < 0.f ? -c : c;
}

// INT3 ("Quantized Cross-Attention ... In-SRAM Dequantization" §3.3: ten
// 3-bit values per 32-bit word) of one D = 128 row: s = fp16(fp32(absmax /
// 3)), code = clamp(RNE(x / s), -3, 3) decided against the exact half-way
// points s/2, 3s/2, 5s/2; element j goes to word j / 10 at bits 3 (j % 10)
// as a 3-bit two's-complement field.  Lane i holds elements 4i..4i+3; lanes
// 0..12 each gather the ten codes of one word by shuffles and store it.
__device__ __forceinline__ int code_of3(float x, float s) {
  const float ax = fabsf(x);
  const float h = 0.5f * s;
  const int m = (ax > h) + (ax >= 3.f * h) + (ax > 5.f * h);
  return x < 0.f ? -m : m;
}

__device__ __forceinline__ void quantize_vals3_warp(const float (&x)[4], uint32_t *dst_words, uint16_t *dst_scale,
                                                    int lane) {
  float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  __half hs = __float2half_rn(__fdiv_rn(am, 3.0f));
  if (__hisinf(hs)) hs = __ushort_as_half(0x7BFF);
  const float s = __half2float(hs);
  uint32_t bytes = 0;  // the lane's four 3-bit fields, one per byte
  if (s > 0.f) {
#pragma unroll
    for (int j = 0; j < 4; ++j) bytes |= (static_cast<uint32_t>(code_of3(x[j], s)) & 7u) << (8 * j);
  }
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const int e = 10 * lane + i;  // element of this lane's word (lanes 0..12 only)
    const uint32_t v = __shfl_sync(0xffffffffu, bytes, (e >> 2) & 31);
    if (e < 128) word |= ((v >> (8 * (e & 3))) & 7u) << (3 * i);
  }
  if (lane < 13) dst_words[lane] = word;
  if (lane == 0) *dst_scale = __half_as_ushort(hs);
}

// INT2 (TurboAttention, arXiv 2412.08585, §3.2's 2-bit heads, in this
// library's per-row symmetric layout) of one D = 128 row: s = fp16(absmax)
// (fp32(absmax / 1) is exact; saturating at 65504), code = clamp(RNE(x / s),
// -1, 1), i.e. +-1 when |x| > s / 2 (a tie at s / 2 goes to the even 0);
// element j goes to word j / 16 at bits 2 (j % 16) as a 2-bit two's-
// complement field.  Lane i holds elements 4i..4i+3, one byte of word i / 4;
// lanes 4k gather the four bytes of word k by shuffles and store it.
__device__ __forceinline__ void quantize_vals2_warp(const float (&x)[4], uint32_t *dst_words, uint16_t *dst_scale,
                                                    int lane) {
  float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  __half hs = __float2half_rn(am);
  if (__hisinf(hs)) hs = __ushort_as_half(0x7BFF);
  const float s = __half2float(hs);
  const float h = 0.5f * s;
  uint32_t byte = 0;  // the lane's four 2-bit fields
  if (s > 0.f) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t f = fabsf(x[j]) > h ? (x[j] < 0.f ? 3u : 1u) : 0u;
      byte |= f << (2 * j);
    }
  }
  const uint32_t b1 = __shfl_down_sync(0xffffffffu, byte, 1);
  const uint32_t b2 = __shfl_down_sync(0xffffffffu, byte, 2);
  const uint32_t b3 = __shfl_down_sync(0xffffffffu, byte, 3);
  if ((lane & 3) == 0) dst_words[lane >> 2] = byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
  if (lane == 0) *dst_scale = __half_as_ushort(hs);
}

}  // namespace qattn
