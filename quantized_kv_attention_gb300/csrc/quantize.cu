// quantize.cu -- quantize-on-append: new K/V rows -> INT4 (INT3, INT2) codes + fp16 scales.
//
// TurboAttention (arXiv 2412.08585) §2.1: each decoding step appends k_t, v_t
// to the cache (prefill appends all prompt rows at once); §2.3: symmetric
// quantization with zero point 0.  "Quantized Cross-Attention ... In-SRAM
// Dequantization" §3.2: 4-bit codes with one FP16 scale per token.
//
// A single HBM pass (D*4 or D*2 bytes read, D/2 + 2 bytes written per INT4
// row), streamed the way the decode kernel streams the cache: a persistent
// grid of two CTAs per SM walks the list of 64-row blocks (K's, then V's);
// in each CTA one producer thread copies its blocks' source rows into a
// 3-deep shared-memory ring with bulk copies (the rows of a block are
// contiguous in k and v unless the cache lists its heads), and 8 consumer
// warps quantize 8 rows each from shared memory and store codes and scales
// to the cache.  INT4 rows take one group of 8 lanes each, so one warp
// instruction works on four rows (quantize_vals_warp4, two rounds, its coding
// arithmetic on packed fp32 pairs); INT3 /
// INT2 rows are quantized one at a time by the whole warp.
#include "internal.h"
#include "ptx.cuh"
#include "quant_row.cuh"

namespace qattn {
namespace {

constexpr int kQWarps = 8;                     // consumer warps
constexpr int kQThreads = (kQWarps + 1) * 32;  // + one producer warp
constexpr int kQWarpRows = 8;                  // rows per consumer warp and block (two rounds of four)
constexpr int kQRows = kQWarps * kQWarpRows;   // rows per block
constexpr int kQCtasPerSm = 2;
constexpr int kQStages = 3;

template <typename T, int D>
struct QCfg {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
  static constexpr int kStageBytes = kQRows * kRowBytes;
  static constexpr int kSmem = kQStages * kStageBytes + 2 * kQStages * 8 + 16 + 128;
};

// The lane's D/32 values of a row held in shared memory at `row`.
template <typename T, int VPL>
__device__ __forceinline__ void lds_row(uint32_t row, int lane, float (&x)[VPL]) {
  if constexpr (sizeof(T) == 4 && VPL == 4) {
    const uint4 u = lds128(row + lane * 16);
    x[0] = __uint_as_float(u.x), x[1] = __uint_as_float(u.y), x[2] = __uint_as_float(u.z), x[3] = __uint_as_float(u.w);
  } else if constexpr (sizeof(T) == 4) {
    const uint2 u = lds64(row + lane * 8);
    x[0] = __uint_as_float(u.x), x[1] = __uint_as_float(u.y);
  } else if constexpr (VPL == 4) {
    const uint2 u = lds64(row + lane * 8);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
  } else {
    uint32_t u;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(u) : "r"(row + lane * 4));
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u));
    x[0] = a.x, x[1] = a.y;
  }
}

// Four consecutive values of type T at shared address p, as floats.
template <typename T>
__device__ __forceinline__ void lds4(uint32_t p, float (&x)[4]) {
  if constexpr (sizeof(T) == 4) {
    const uint4 u = lds128(p);
    x[0] = __uint_as_float(u.x), x[1] = __uint_as_float(u.y), x[2] = __uint_as_float(u.z), x[3] = __uint_as_float(u.w);
  } else {
    const uint2 u = lds64(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
  }
}

// Cache row of source row i of (sequence b, cache head h), bh = b * Hkv + h,
// or -1 when the row is not written: its position is past the capacity or in
// no page, its page is missing (flagged) or the head map does not name the
// head (flagged).  Only a lane with `flag` set raises the flags.
__device__ __forceinline__ int64_t dest_row(const KvView &cache, const int32_t *__restrict__ start_pos, int b,
                                            int h, int64_t bh, int i, bool flag, uint32_t *err) {
  if (model_head(cache.head_map, cache.model_hkv, h) < 0) {
    if (flag && err) atomicOr(err, kFlagBadHead);
    return -1;
  }
  const int64_t pos = static_cast<int64_t>(start_pos ? __ldg(start_pos + b) : 0) + i;
  if (cache.page_table == nullptr) return pos >= 0 && pos < cache.capacity ? bh * cache.capacity + pos : -1;
  if (pos < 0 || pos / kPage >= cache.max_pages) return -1;
  const int page = __ldg(cache.page_table + static_cast<int64_t>(b) * cache.max_pages + pos / kPage);
  if (page >= 0 && page < cache.num_pages) return (static_cast<int64_t>(page) * cache.hkv + h) * kPage + (pos % kPage);
  if (flag && err) atomicOr(err, kFlagBadPage);
  return -1;
}

template <typename T, int D, bool kInt4>
__global__ void __launch_bounds__(kQThreads, kQCtasPerSm)
    quantize_kv_kernel(const T *__restrict__ k, const T *__restrict__ v, int batch, int n,
                       const int32_t *__restrict__ start_pos, KvView cache, uint32_t *err) {
  using C = QCfg<T, D>;
  constexpr int VPL = D / 32;  // values per lane
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kQStages * C::kStageBytes);
  uint64_t *empty = full + kQStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kQStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;  // per tensor
  const int64_t per_tensor = (rows + kQRows - 1) / kQRows;            // blocks per tensor
  const int64_t blocks = 2 * per_tensor;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kQWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kQWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      for (int64_t blk = blockIdx.x; blk < blocks; blk += gridDim.x, ++it) {
        const int s = it % kQStages;
        if (it >= kQStages &&
            !mbar_wait(smem_u32(empty + s), ((it / kQStages) & 1) ^ 1, err, *abort_flag ? kDrainCycles : kWaitCycles)) {
          *abort_flag = 1;
          break;
        }
        const bool is_v = blk >= per_tensor;
        const int64_t r0 = (is_v ? blk - per_tensor : blk) * kQRows;
        const int nr = static_cast<int>(min(static_cast<int64_t>(kQRows), rows - r0));
        const T *base = is_v ? v : k;
        const uint32_t dst = smem_u32(smem + s * C::kStageBytes);
        const uint32_t bar = smem_u32(full + s);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr * C::kRowBytes));
        if (cache.head_map == nullptr) {
          // rows r0.. are source rows r0.. of [batch, Hkv, n, D]: one copy
          bulk_g2s(dst, base + r0 * D, static_cast<uint32_t>(nr * C::kRowBytes), bar);
        } else {
          // a listed cache reads the model's rows: one copy per run of rows
          // of one (sequence, head); a head the map does not name loads
          // model head 0 (its rows are flagged and skipped by the consumers)
          int i = static_cast<int>(r0 % n);
          int64_t bh = r0 / n;
          for (int j = 0; j < nr;) {
            const int run = min(nr - j, n - i);
            const int h = static_cast<int>(bh % cache.hkv), b = static_cast<int>(bh / cache.hkv);
            const int mh = max(model_head(cache.head_map, cache.model_hkv, h), 0);
            const T *src = base + ((static_cast<int64_t>(b) * cache.model_hkv + mh) * n + i) * D;
            bulk_g2s(dst + j * C::kRowBytes, src, static_cast<uint32_t>(run * C::kRowBytes), bar);
            j += run, i = 0, ++bh;
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // (b, h, i) of the warp's first row: one pair of divisions when the CTA
  // enters a tensor, then a step of gridDim.x blocks by additions
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kQRows;  // rows between a CTA's blocks
  const int64_t step_bh = stride / n;
  const int step_i = static_cast<int>(stride - step_bh * n);
  const int step_h = static_cast<int>(step_bh % cache.hkv);
  const int step_b = static_cast<int>(step_bh / cache.hkv);
  int64_t bh = 0, sp = 0;  // sp: start_pos[sp_b]
  int i = 0, h = 0, b = 0, tensor = -1, sp_b = -1;
  int it = 0;
  for (int64_t blk = blockIdx.x; blk < blocks; blk += gridDim.x, ++it) {
    const int s = it % kQStages;
    const bool got = mbar_wait(smem_u32(full + s), (it / kQStages) & 1, err, *abort_flag ? kDrainCycles : kWaitCycles);
    if (!got) *abort_flag = 1;
    const bool is_v = blk >= per_tensor;
    const int64_t r0 = (is_v ? blk - per_tensor : blk) * kQRows;
    uint8_t *codes = is_v ? cache.v_codes : cache.k_codes;
    uint16_t *scales = is_v ? cache.v_scales : cache.k_scales;
    const int64_t rw = r0 + warp * kQWarpRows;
    if (tensor != static_cast<int>(is_v)) {
      tensor = is_v;
      if (rows < (int64_t(1) << 31)) {
        const uint32_t q = static_cast<uint32_t>(rw) / static_cast<uint32_t>(n);
        bh = q, i = static_cast<int>(static_cast<uint32_t>(rw) - q * static_cast<uint32_t>(n));
      } else {
        bh = rw / n, i = static_cast<int>(rw - bh * n);
      }
      h = static_cast<int>(bh % cache.hkv), b = static_cast<int>(bh / cache.hkv);
    } else {
      i += step_i, bh += step_bh, h += step_h, b += step_b;
      if (i >= n) i -= n, ++bh, ++h;
      if (h >= cache.hkv) h -= cache.hkv, ++b;
    }
    // the warp's rows of one (sequence, head) going to consecutive cache rows
    // (contiguous, or inside one page): one destination for all of them
    int64_t span_row = -1;
    if (got && rw + kQWarpRows - 1 < rows && i + kQWarpRows - 1 < n && cache.head_map == nullptr) {
      if (b != sp_b) sp_b = b, sp = start_pos ? __ldg(start_pos + b) : 0;
      const int64_t pos = sp + i;
      if (cache.page_table == nullptr) {
        if (pos >= 0 && pos + kQWarpRows - 1 < cache.capacity) span_row = bh * cache.capacity + pos;
      } else if (pos >= 0 && pos % kPage + kQWarpRows - 1 < kPage && pos / kPage < cache.max_pages) {
        const int page = __ldg(cache.page_table + static_cast<int64_t>(b) * cache.max_pages + pos / kPage);
        if (page >= 0 && page < cache.num_pages)
          span_row = (static_cast<int64_t>(page) * cache.hkv + h) * kPage + (pos % kPage);
      }
      // otherwise row by row below (which flags a missing page)
    }
    const uint32_t stage = smem_u32(smem + s * C::kStageBytes + warp * kQWarpRows * C::kRowBytes);
    if constexpr (kInt4) {
      // round u: lane group g = lane / 8 takes the warp's row 4u + g
      const int g = lane >> 3, l = lane & 7;
#pragma unroll 1
      for (int u = 0; u < kQWarpRows / 4; ++u) {
        const int wr = 4 * u + g;  // the group's row within the warp's rows
        int64_t dst = span_row >= 0 ? span_row + wr : -1;
        if (span_row < 0 && got && rw + wr < rows) {
          int64_t bhg = bh;
          int ig = i, hg = h, bg = b;
          for (int r = 0; r < wr; ++r)
            if (++ig == n) {
              ig = 0, ++bhg;
              if (++hg == cache.hkv) hg = 0, ++bg;
            }
          dst = dest_row(cache, start_pos, bg, hg, bhg, ig, l == 0, err);
        }
        constexpr int NC = D / 32;  // chunks of 32 values
        float x[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int cc = (c + g) & (NC - 1);
          if (dst >= 0)
            lds4<T>(stage + wr * C::kRowBytes + (cc * 32 + 4 * l) * static_cast<int>(sizeof(T)), x[c]);
          else
            x[c][0] = x[c][1] = x[c][2] = x[c][3] = 0.f;
        }
        quantize_vals_warp4<D>(x, dst >= 0 ? codes + dst * (D / 2) : nullptr, scales + (dst >= 0 ? dst : 0), lane);
      }
    } else {
      // INT3 / INT2 (D = 128): the warp quantizes its rows one by one
      const int tb = cache.bits == 3 ? 52 : 32;  // code bytes per row
      int64_t bh_r = bh;
      int i_r = i, h_r = h, b_r = b;
#pragma unroll 1
      for (int r = 0; r < kQWarpRows; ++r, ++i_r) {
        if (i_r == n) {
          i_r = 0, ++bh_r;
          if (++h_r == cache.hkv) h_r = 0, ++b_r;
        }
        int64_t dst = span_row >= 0 ? span_row + r : -1;
        if (span_row < 0 && got && rw + r < rows) dst = dest_row(cache, start_pos, b_r, h_r, bh_r, i_r, lane == 0, err);
        if (dst < 0) continue;  // warp-uniform
        float x[VPL];
        lds_row<T, VPL>(stage + r * C::kRowBytes, lane, x);
        if (cache.bits == 3)
          quantize_vals3_warp(x, reinterpret_cast<uint32_t *>(codes + dst * tb), scales + dst, lane);
        else
          quantize_vals2_warp(x, reinterpret_cast<uint32_t *>(codes + dst * tb), scales + dst, lane);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }
}

template <typename T, int D, bool kInt4>
cudaError_t launch_t(const void *k, const void *v, int batch, int n, const int32_t *start_pos,
                     const KvView &cache, uint32_t *err, int sms, cudaStream_t stream) {
  using C = QCfg<T, D>;
  static bool configured = false;  // per-function attribute, set once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(quantize_kv_kernel<T, D, kInt4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = 2 * ((rows + kQRows - 1) / kQRows);
  const int64_t grid = min(blocks, static_cast<int64_t>(kQCtasPerSm * (sms > 0 ? sms : 1)));
  quantize_kv_kernel<T, D, kInt4><<<static_cast<unsigned>(grid), kQThreads, C::kSmem, stream>>>(
      static_cast<const T *>(k), static_cast<const T *>(v), batch, n, start_pos, cache, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void *k, const void *v, bool fp16_in, int batch, int n,
                            const int32_t *start_pos, const KvView &cache, uint32_t *err, int sms,
                            cudaStream_t stream) {
  if (cache.bits != 4)  // INT3 / INT2: D = 128 (checked by the caller)
    return fp16_in ? launch_t<__half, 128, false>(k, v, batch, n, start_pos, cache, err, sms, stream)
                   : launch_t<float, 128, false>(k, v, batch, n, start_pos, cache, err, sms, stream);
  if (cache.head_dim == 128)
    return fp16_in ? launch_t<__half, 128, true>(k, v, batch, n, start_pos, cache, err, sms, stream)
                   : launch_t<float, 128, true>(k, v, batch, n, start_pos, cache, err, sms, stream);
  return fp16_in ? launch_t<__half, 64, true>(k, v, batch, n, start_pos, cache, err, sms, stream)
                 : launch_t<float, 64, true>(k, v, batch, n, start_pos, cache, err, sms, stream);
}

}  // namespace qattn
