// quantize.cu -- quantize-on-append: new K/V rows -> INT4 codes + fp16 scales.
//
// TurboAttention (arXiv 2412.08585) §2.1: each decoding step appends k_t, v_t
// to the cache (prefill appends all prompt rows at once); §2.3: symmetric
// quantization with zero point 0.  "Quantized Cross-Attention ... In-SRAM
// Dequantization" §3.2: 4-bit codes with one FP16 scale per token.
//
// One warp per row of D values; the kernel is a single HBM pass (read D*4 or
// D*2 bytes, write D/2 + 2 bytes per row).  The rounding of each code is
// decided by exact comparisons with the half-way points (k + 1/2) * s, which
// are exact in fp32 (s has 11 significant bits, 2k + 1 at most 4), so the
// result equals round-half-even of the exact quotient x / s.
#include "internal.h"
#include "ptx.cuh"

namespace qattn {
namespace {

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

template <typename T, int D>
__global__ void __launch_bounds__(256)
    quantize_kv_kernel(const T *__restrict__ k, const T *__restrict__ v, int batch, int n,
                       const int32_t *__restrict__ start_pos, KvView cache, uint32_t *err) {
  constexpr int VPL = D / 32;  // values per lane
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;
  if (row >= rows) return;
  const bool is_v = blockIdx.y != 0;
  const T *src = (is_v ? v : k) + row * D + lane * VPL;

  const int i = static_cast<int>(row % n);
  const int64_t bh = row / n;
  const int h = static_cast<int>(bh % cache.hkv);
  const int b = static_cast<int>(bh / cache.hkv);
  const int64_t pos = static_cast<int64_t>(start_pos ? __ldg(start_pos + b) : 0) + i;

  int64_t dst_row = -1;  // row index in the destination cache
  if (cache.page_table == nullptr) {
    if (pos >= 0 && pos < cache.capacity) dst_row = bh * cache.capacity + pos;
  } else if (pos >= 0 && pos / kPage < cache.max_pages) {
    const int page = __ldg(cache.page_table + static_cast<int64_t>(b) * cache.max_pages + pos / kPage);
    if (page >= 0 && page < cache.num_pages)
      dst_row = (static_cast<int64_t>(page) * cache.hkv + h) * kPage + (pos % kPage);
    else if (lane == 0 && err)
      atomicOr(err, kFlagBadPage);
  }
  if (dst_row < 0) return;  // warp-uniform

  float x[VPL];
  RowLoad<T, VPL>::load(src, x);
  float am = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) am = fmaxf(am, fabsf(x[j]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));

  // s = fp16(fp32(am / 7)), both roundings to nearest even; saturate at 65504.
  __half hs = __float2half_rn(__fdiv_rn(am, 7.0f));
  if (__hisinf(hs)) hs = __ushort_as_half(0x7BFF);
  const float s = __half2float(hs);

  uint32_t packed = 0;
  if (s > 0.f) {
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      packed |= static_cast<uint32_t>(code_of(x[j], s) & 0xF) << (4 * j);
  }
  uint8_t *codes = is_v ? cache.v_codes : cache.k_codes;
  uint16_t *scales = is_v ? cache.v_scales : cache.k_scales;
  uint8_t *dst = codes + dst_row * (D / 2) + lane * (VPL / 2);
  if constexpr (VPL == 4)
    *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
  else
    *dst = static_cast<uint8_t>(packed);
  if (lane == 0) scales[dst_row] = __half_as_ushort(hs);
}

template <typename T, int D>
cudaError_t launch_t(const void *k, const void *v, int batch, int n, const int32_t *start_pos,
                     const KvView &cache, uint32_t *err, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;
  if (rows == 0) return cudaSuccess;
  constexpr int kWarps = 8;
  dim3 grid(static_cast<unsigned>((rows + kWarps - 1) / kWarps), 2);
  quantize_kv_kernel<T, D><<<grid, kWarps * 32, 0, stream>>>(
      static_cast<const T *>(k), static_cast<const T *>(v), batch, n, start_pos, cache, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void *k, const void *v, bool fp16_in, int batch, int n,
                            const int32_t *start_pos, const KvView &cache, uint32_t *err,
                            cudaStream_t stream) {
  if (cache.head_dim == 128)
    return fp16_in ? launch_t<__half, 128>(k, v, batch, n, start_pos, cache, err, stream)
                   : launch_t<float, 128>(k, v, batch, n, start_pos, cache, err, stream);
  return fp16_in ? launch_t<__half, 64>(k, v, batch, n, start_pos, cache, err, stream)
                 : launch_t<float, 64>(k, v, batch, n, start_pos, cache, err, stream);
}

}  // namespace qattn
