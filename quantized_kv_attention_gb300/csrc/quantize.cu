// quantize.cu -- quantize-on-append: new K/V rows -> INT4 (INT3, INT2) codes + fp16 scales.
//
// TurboAttention (arXiv 2412.08585) §2.1: each decoding step appends k_t, v_t
// to the cache (prefill appends all prompt rows at once); §2.3: symmetric
// quantization with zero point 0.  "Quantized Cross-Attention ... In-SRAM
// Dequantization" §3.2: 4-bit codes with one FP16 scale per token.
//
// One warp per row of D values (quantize_row_warp); the kernel is a single
// HBM pass (read D*4 or D*2 bytes, write D/2 + 2 bytes per row).
#include "internal.h"
#include "ptx.cuh"
#include "quant_row.cuh"

namespace qattn {
namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256)
    quantize_kv_kernel(const T *__restrict__ k, const T *__restrict__ v, int batch, int n,
                       const int32_t *__restrict__ start_pos, KvView cache, uint32_t *err) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;
  if (row >= rows) return;
  const bool is_v = blockIdx.y != 0;

  const int i = static_cast<int>(row % n);
  const int64_t bh = row / n;
  const int h = static_cast<int>(bh % cache.hkv);
  const int b = static_cast<int>(bh / cache.hkv);
  // the source rows are the model's: cache head h reads model head head_map[h]
  const int mh = model_head(cache.head_map, cache.model_hkv, h);
  if (mh < 0) {  // warp-uniform
    if (lane == 0 && err) atomicOr(err, kFlagBadHead);
    return;
  }
  const T *src = (is_v ? v : k) + ((static_cast<int64_t>(b) * cache.model_hkv + mh) * n + i) * D;
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

  uint8_t *codes = is_v ? cache.v_codes : cache.k_codes;
  uint16_t *scales = is_v ? cache.v_scales : cache.k_scales;
  if constexpr (D == 128) {
    if (cache.bits == 3) {  // 13 words per row
      quantize_row3_warp<T>(src, reinterpret_cast<uint32_t *>(codes + dst_row * 52), scales + dst_row, lane);
      return;
    }
    if (cache.bits == 2) {  // 8 words per row
      quantize_row2_warp<T>(src, reinterpret_cast<uint32_t *>(codes + dst_row * 32), scales + dst_row, lane);
      return;
    }
  }
  quantize_row_warp<T, D>(src, codes + dst_row * (D / 2), scales + dst_row, lane);
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
