// quant_row.cuh -- quantization of one K or V row (D values) by one warp,
// shared by the append kernel and the fused append + decode step so that
// both write the same bits.
//
// TurboAttention (arXiv 2412.08585) §2.3: symmetric quantization, zero point
// 0; "Quantized Cross-Attention ... In-SRAM Dequantization" §3.2: 4-bit codes
// with one FP16 scale per token.  s = fp16(fp32(absmax / 7)), both roundings
// to nearest even, saturating at 65504; code = round-half-even(x / s) clamped
// to [-7, 7], decided by exact comparisons with the half-way points
// (k + 1/2) s, which are exact in fp32 (s has 11 significant bits, 2k + 1 at
// most 4 bits), so the result equals rounding of the exact quotient.
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

  uint32_t packed = 0;
  if (s > 0.f) {
#pragma unroll
    for (int j = 0; j < VPL; ++j) packed |= static_cast<uint32_t>(code_of(x[j], s) & 0xF) << (4 * j);
  }
  uint8_t *dst = dst_codes + lane * (VPL / 2);
  if constexpr (VPL == 4)
    *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
  else
    *dst = static_cast<uint8_t>(packed);
  if (lane == 0) *dst_scale = __half_as_ushort(hs);
  return hs;
}

// quantize_vals_warp for N rows at once (the same arithmetic, so the same
// bits), phase by phase across the rows so that their shuffle reductions and
// divisions overlap; a row whose dst_codes is null is computed but not stored.
template <int D, int N>
__device__ __forceinline__ void quantize_vals_warp_n(const float (&x)[N][D / 32], uint8_t *const (&dst_codes)[N],
                                                     uint16_t *const (&dst_scale)[N], int lane) {
  constexpr int VPL = D / 32;
  float am[N];
#pragma unroll
  for (int r = 0; r < N; ++r) {
    am[r] = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) am[r] = fmaxf(am[r], fabsf(x[r][j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < N; ++r) am[r] = fmaxf(am[r], __shfl_xor_sync(0xffffffffu, am[r], o));
  __half hs[N];
#pragma unroll
  for (int r = 0; r < N; ++r) {
    hs[r] = __float2half_rn(__fdiv_rn(am[r], 7.0f));
    if (__hisinf(hs[r])) hs[r] = __ushort_as_half(0x7BFF);
  }
#pragma unroll
  for (int r = 0; r < N; ++r) {
    const float s = __half2float(hs[r]);
    uint32_t packed = 0;
    if (s > 0.f) {
#pragma unroll
      for (int j = 0; j < VPL; ++j) packed |= static_cast<uint32_t>(code_of(x[r][j], s) & 0xF) << (4 * j);
    }
    if (dst_codes[r] != nullptr) {
      uint8_t *dst = dst_codes[r] + lane * (VPL / 2);
      if constexpr (VPL == 4)
        *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
      else
        *dst = static_cast<uint8_t>(packed);
      if (lane == 0) *dst_scale[r] = __half_as_ushort(hs[r]);
    }
  }
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
