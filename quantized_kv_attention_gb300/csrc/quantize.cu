// quantize.cu -- quantize-on-append: new K/V rows -> INT4 (INT3, INT2) codes + fp16 scales.
//
// TurboAttention (arXiv 2412.08585) §2.1: each decoding step appends k_t, v_t
// to the cache (prefill appends all prompt rows at once); §2.3: symmetric
// quantization with zero point 0.  "Quantized Cross-Attention ... In-SRAM
// Dequantization" §3.2: 4-bit codes with one FP16 scale per token.
//
// A single HBM pass (D*4 or D*2 bytes read, D/2 + 2 bytes written per INT4
// row), streamed the way the decode kernel streams the cache: a persistent
// grid of four CTAs per SM walks the list of 32-row blocks (K's, then V's);
// in each CTA one producer thread copies its blocks' source rows into a
// 3-deep shared-memory ring with bulk copies (the rows of a block are
// contiguous in k and v unless the cache lists its heads), and 8 consumer
// warps quantize 4 rows each from shared memory (quantize_vals_warp_n, the
// four rows' reductions interleaved; the INT3 / INT2 forms row by row) and
// store codes and scales to the cache.  The work is bound by instruction
// issue (the exact round-half-even decision per value), so the grid keeps
// 32 consumer warps per SM.
#include "internal.h"
#include "ptx.cuh"
#include "quant_row.cuh"

namespace qattn {
namespace {

constexpr int kQWarps = 8;                     // consumer warps
constexpr int kQThreads = (kQWarps + 1) * 32;  // + one producer warp
constexpr int kQRows = 32;                     // rows per block (4 per consumer warp)
constexpr int kQCtasPerSm = 4;                 // quantizing is issue-bound: many warps per SM
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

template <typename T, int D>
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
  int it = 0;
  for (int64_t blk = blockIdx.x; blk < blocks; blk += gridDim.x, ++it) {
    const int s = it % kQStages;
    const bool got = mbar_wait(smem_u32(full + s), (it / kQStages) & 1, err, *abort_flag ? kDrainCycles : kWaitCycles);
    if (!got) *abort_flag = 1;
    const bool is_v = blk >= per_tensor;
    const int64_t r0 = (is_v ? blk - per_tensor : blk) * kQRows;
    uint8_t *codes = is_v ? cache.v_codes : cache.k_codes;
    uint16_t *scales = is_v ? cache.v_scales : cache.k_scales;
    // (b, h, i) of the warp's first row by one pair of divisions (32-bit
    // when the row count allows), then stepped row by row
    const int64_t rw = r0 + warp * 4;
    int64_t bh;
    int i;
    if (rows < (int64_t(1) << 31)) {
      const uint32_t q = static_cast<uint32_t>(rw) / static_cast<uint32_t>(n);
      bh = q, i = static_cast<int>(static_cast<uint32_t>(rw) - q * static_cast<uint32_t>(n));
    } else {
      bh = rw / n, i = static_cast<int>(rw - bh * n);
    }
    int h = static_cast<int>(static_cast<uint32_t>(bh) % static_cast<uint32_t>(cache.hkv));
    int b = static_cast<int>(static_cast<uint32_t>(bh) / static_cast<uint32_t>(cache.hkv));
    // the warp's 4 rows: destinations and values first, then (INT4) one
    // quantization of all four with their reductions interleaved
    uint8_t *dc[4];
    uint16_t *ds[4];
    float x[4][VPL];
#pragma unroll
    for (int r = 0; r < 4; ++r, ++i) {
      if (i == n) {
        i = 0, ++bh;
        if (++h == cache.hkv) h = 0, ++b;
      }
      dc[r] = nullptr, ds[r] = nullptr;
      const int64_t row = rw + r;
      if (got && row < rows) {
        if (model_head(cache.head_map, cache.model_hkv, h) < 0) {
          if (lane == 0 && err) atomicOr(err, kFlagBadHead);
        } else {
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
          if (dst_row >= 0) {
            const int tb = cache.bits == 3 ? 52 : cache.bits == 2 ? 32 : D / 2;  // code bytes per row
            dc[r] = codes + dst_row * tb, ds[r] = scales + dst_row;
          }
        }
      }
      if (dc[r] != nullptr)
        lds_row<T, VPL>(smem_u32(smem + s * C::kStageBytes + (warp * 4 + r) * C::kRowBytes), lane, x[r]);
      else
#pragma unroll
        for (int j = 0; j < VPL; ++j) x[r][j] = 0.f;
    }
    if (D == 128 && cache.bits != 4) {
      if constexpr (D == 128) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (dc[r] == nullptr) continue;  // warp-uniform
          if (cache.bits == 3)
            quantize_vals3_warp(x[r], reinterpret_cast<uint32_t *>(dc[r]), ds[r], lane);
          else
            quantize_vals2_warp(x[r], reinterpret_cast<uint32_t *>(dc[r]), ds[r], lane);
        }
      }
    } else {
      quantize_vals_warp_n<D, 4>(x, dc, ds, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }
}

template <typename T, int D>
cudaError_t launch_t(const void *k, const void *v, int batch, int n, const int32_t *start_pos,
                     const KvView &cache, uint32_t *err, int sms, cudaStream_t stream) {
  using C = QCfg<T, D>;
  static bool configured = false;  // per-function attribute, set once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(quantize_kv_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t rows = static_cast<int64_t>(batch) * cache.hkv * n;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = 2 * ((rows + kQRows - 1) / kQRows);
  const int64_t grid = min(blocks, static_cast<int64_t>(kQCtasPerSm * (sms > 0 ? sms : 1)));
  quantize_kv_kernel<T, D><<<static_cast<unsigned>(grid), kQThreads, C::kSmem, stream>>>(
      static_cast<const T *>(k), static_cast<const T *>(v), batch, n, start_pos, cache, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void *k, const void *v, bool fp16_in, int batch, int n,
                            const int32_t *start_pos, const KvView &cache, uint32_t *err, int sms,
                            cudaStream_t stream) {
  if (cache.head_dim == 128)
    return fp16_in ? launch_t<__half, 128>(k, v, batch, n, start_pos, cache, err, sms, stream)
                   : launch_t<float, 128>(k, v, batch, n, start_pos, cache, err, sms, stream);
  return fp16_in ? launch_t<__half, 64>(k, v, batch, n, start_pos, cache, err, sms, stream)
                 : launch_t<float, 64>(k, v, batch, n, start_pos, cache, err, sms, stream);
}

}  // namespace qattn
