// flashq.cu -- a FlashQ-style decode buffer in front of the INT4 cache.
//
// TurboAttention (arXiv 2412.08585) §3.3: newly decoded K/V rows wait in a
// buffer of 64 rows, quantized to 8 bits (§3.2, Equation 9's symmetric first
// stage) with one universal scale and outliers clamped, so that buffered rows
// never need re-quantizing; a full buffer is compressed into the low-bit
// cache.  Here the cache is the per-row INT4 format of the rest of the
// library, and the universal scale of a (sequence, kv-head) and tensor is
// u = fp16(fp32(R / 127)), R = 7 x the largest row scale of its cached rows
// (their max |x^|), raised at every flush; while R is 0 each appended row
// sets it to its own absmax.
//
//   flashq_init    R, u from the cached rows; empty buffers
//   flashq_append  one new K and V row per (sequence, kv-head) -> int8 codes
//                  c = clamp(RNE(x / u), -127, 127) in the next buffer slot
//   flashq_attend  attention of q over the buffered rows (x~ = c * u),
//                  merged by log-sum-exp into the O and lse a qattn_decode
//                  over the cached rows left in out / lse
//   flashq_flush   a full buffer -> 64 INT4 rows in the cache (the INT4
//                  codec of quant_row.cuh on x~), R and u raised, buffer empty
//
// All four are small (the buffer holds at most 64 rows per head) and run one
// CTA per sequence or per (sequence, kv-head); none waits on another CTA.
#include <math.h>

#include "../../include/qattn.h"
#include "internal.h"
#include "ptx.cuh"
#include "quant_row.cuh"

namespace qattn {
namespace {

constexpr uint32_t kFlagBufferFull = 8u;  // an append found a full buffer (row dropped)
constexpr int kNb = 64;                   // buffer rows

// Cache row of token `pos` of (b, h): contiguous or through the page table;
// -1 past the cache or in a missing page.
__device__ __forceinline__ int64_t cache_row(const KvView &c, int b, int h, int64_t pos) {
  if (!c.page_table) return pos < c.capacity ? (static_cast<int64_t>(b) * c.hkv + h) * c.capacity + pos : -1;
  if (pos / kPage >= c.max_pages) return -1;
  const int page = __ldg(c.page_table + static_cast<int64_t>(b) * c.max_pages + pos / kPage);
  if (page < 0 || page >= c.num_pages) return -1;
  return (static_cast<int64_t>(page) * c.hkv + h) * kPage + pos % kPage;
}

// Grid (batch * Hkv * 2), 256 threads: R = 7 * max scale of the first
// cache_lens[b] rows of (b, h) for K (y even) or V; u from R.
__global__ void __launch_bounds__(256) flashq_init_kernel(FlashqView f, KvView c, const int32_t *cache_lens,
                                                          int batch) {
  const int idx = blockIdx.x;
  const int t = idx & 1, bh = idx >> 1;
  const int b = bh / c.hkv, h = bh % c.hkv;
  const uint16_t *sc = t ? c.v_scales : c.k_scales;
  const int64_t n = max(0, __ldg(cache_lens + b));
  float mx = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t row = cache_row(c, b, h, i);
    if (row >= 0) mx = fmaxf(mx, __half2float(__ushort_as_half(sc[row])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, wmax[w]);
    const float r = 7.f * mx;  // exact: an 11-bit scale times 7
    (t ? f.v_range : f.k_range)[bh] = r;
    (t ? f.v_scale : f.k_scale)[bh] = __half_as_ushort(universal_scale(r));
    if (t == 0 && h == 0) f.count[b] = 0;
  }
}

// Grid batch; warp w takes rows w, w + nwarps, ... of the 2 * Hkv (head,
// tensor) rows of its sequence; lane i holds elements 4i..4i+3 (D = 128) or
// 2i, 2i+1 (D = 64).
template <typename T, int D>
__global__ void __launch_bounds__(1024) flashq_append_kernel(const T *__restrict__ k, const T *__restrict__ v,
                                                             FlashqView f, int batch, uint32_t *err) {
  constexpr int VPL = D / 32;
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int slot = f.count[b];
  __syncthreads();  // every warp has read the count before it moves
  if (slot >= kNb) {
    if (threadIdx.x == 0) atomicOr(err, kFlagBufferFull);
    return;
  }
  for (int r = warp; r < 2 * f.hkv; r += nwarps) {
    const int h = r >> 1, t = r & 1;
    const int64_t bh = static_cast<int64_t>(b) * f.hkv + h;
    float x[VPL];
    RowLoad<T, VPL>::load((t ? v : k) + bh * D + lane * VPL, x);
    float am = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) am = fmaxf(am, fabsf(x[j]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    float *range = t ? f.v_range : f.k_range;
    float rr = range[bh];
    if (rr == 0.f) {  // no range yet: this row sets it
      rr = am;
      __syncwarp();
      if (lane == 0) range[bh] = rr;
    }
    const __half uh = universal_scale(rr);
    if (lane == 0) (t ? f.v_scale : f.k_scale)[bh] = __half_as_ushort(uh);
    const float u = __half2float(uh);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < VPL; ++j) packed |= (static_cast<uint32_t>(code8(x[j], u)) & 0xFFu) << (8 * j);
    int8_t *dst = (t ? f.v_codes : f.k_codes) + (bh * kNb + slot) * D + lane * VPL;
    if constexpr (VPL == 4)
      *reinterpret_cast<uint32_t *>(dst) = packed;
    else
      *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
  }
  __syncthreads();
  if (threadIdx.x == 0) f.count[b] = slot + 1;
}

// Grid (batch * Hq), 128 threads: one query row (sequence b, query head g of
// kv-head h = g / G).  S_t = q . x~_K,t * scale (log2 units) over the n
// buffered rows, p = 2^(S - m_b), O_b = sum p x~_V / l_b, lse_b =
// (m_b + log2 l_b) ln 2; then merged with the (O_c, lse_c) already in out /
// lse: L = log(e^lse_c + e^lse_b), O = e^(lse_c - L) O_c + e^(lse_b - L) O_b.
// Launched as a programmatic dependent: the buffer part is done before the
// wait -- the kernels that may still run then are this library's decode,
// merge and combine kernels, which never write the buffer (the append
// releases no dependent early) -- and out / lse after it.
template <int D>
__global__ void __launch_bounds__(128) flashq_attend_kernel(const uint16_t *__restrict__ q, FlashqView f, int batch,
                                                            int hq, float scale_log2, uint16_t *out, float *lse) {
  constexpr int VPL = D / 32;
  const int64_t row = blockIdx.x;  // b * hq + query head
  const int b = static_cast<int>(row / hq), G = hq / f.hkv;
  const int64_t bh = static_cast<int64_t>(b) * f.hkv + static_cast<int>(row % hq) / G;
  const int n = min(f.count[b], kNb);
  if (n <= 0) return;
  __shared__ float qs[D];
  __shared__ float ps[kNb];
  __shared__ int8_t ck[kNb][D], cv[kNb][D];
  __shared__ float mls[3];  // m_b, l_b, lse_c
  const float uk = __half2float(__ushort_as_half(f.k_scale[bh])), uv = __half2float(__ushort_as_half(f.v_scale[bh]));
  for (int i = threadIdx.x; i < D; i += blockDim.x) qs[i] = __half2float(__ushort_as_half(q[row * D + i]));
  for (int i = threadIdx.x; i < n * D / 16; i += blockDim.x) {
    reinterpret_cast<uint4 *>(&ck[0][0])[i] = reinterpret_cast<const uint4 *>(f.k_codes + bh * kNb * D)[i];
    reinterpret_cast<uint4 *>(&cv[0][0])[i] = reinterpret_cast<const uint4 *>(f.v_codes + bh * kNb * D)[i];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < n; t += blockDim.x >> 5) {  // scores: a warp per buffered row
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) acc = fmaf(qs[VPL * lane + j], static_cast<float>(ck[t][VPL * lane + j]), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) ps[t] = acc * uk * scale_log2;
  }
  __syncthreads();
  if (warp == 0) {  // softmax of the row
    float m = -INFINITY;
    for (int t = lane; t < n; t += 32) m = fmaxf(m, ps[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int t = lane; t < n; t += 32) {
      const float p = exp2f(ps[t] - m);
      ps[t] = p;
      l += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) mls[0] = m, mls[1] = l;
  }
  __syncthreads();
  constexpr int kCols = (D + 127) / 128;  // columns of O a thread keeps
  float ob[kCols];
#pragma unroll
  for (int k = 0; k < kCols; ++k) {  // O_b
    const int d = threadIdx.x + 128 * k;
    float acc = 0.f;
    if (d < D)
      for (int t = 0; t < n; ++t) acc = fmaf(ps[t], static_cast<float>(cv[t][d]), acc);
    ob[k] = acc * uv / mls[1];
  }
  pdl_wait();  // out and lse of the cache part come from the preceding kernel
  if (threadIdx.x == 0) mls[2] = lse[row];
  __syncthreads();  // lse_c is read before it is overwritten below
  const float lse_b = (mls[0] + log2f(mls[1])) * 0.69314718055994531f, lse_c = mls[2];
  const float mx = fmaxf(lse_c, lse_b);
  const float wc = expf(lse_c - mx), wb = expf(lse_b - mx);  // e^-inf = 0 for an empty cache part
  const float z = wc + wb;
#pragma unroll
  for (int k = 0; k < kCols; ++k) {  // the merge
    const int d = threadIdx.x + 128 * k;
    if (d >= D) continue;
    const float oc = __half2float(__ushort_as_half(out[row * D + d]));
    out[row * D + d] = __half_as_ushort(__float2half_rn((wc * oc + wb * ob[k]) / z));
  }
  if (threadIdx.x == 0) lse[row] = mx + logf(z);
}

// Grid batch, 512 threads: a sequence whose buffer is full moves its 64 rows
// (all kv-heads, K and V) into the INT4 cache at positions cache_lens[b] ..
// + 63, raises R and u, and empties the buffer.
template <int D>
__global__ void __launch_bounds__(512) flashq_flush_kernel(FlashqView f, KvView c, const int32_t *cache_lens,
                                                           int batch, uint32_t *err) {
  constexpr int VPL = D / 32;
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (f.count[b] < kNb) return;  // uniform across the block
  __shared__ float smax[2 * 64];  // [head][tensor]: largest new row scale (Hkv <= 64)
  for (int i = threadIdx.x; i < 2 * f.hkv; i += blockDim.x) smax[i] = 0.f;
  __syncthreads();
  const int64_t base = __ldg(cache_lens + b);
  for (int r = warp; r < 2 * f.hkv * kNb; r += nwarps) {
    const int i = r % kNb, ht = r / kNb, h = ht >> 1, t = ht & 1;
    const int64_t bh = static_cast<int64_t>(b) * f.hkv + h;
    const float u = __half2float(__ushort_as_half((t ? f.v_scale : f.k_scale)[bh]));
    const int8_t *src = (t ? f.v_codes : f.k_codes) + (bh * kNb + i) * D + lane * VPL;
    float x[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) x[j] = static_cast<float>(src[j]) * u;  // exact: 8 x 11 bits
    const int64_t row = cache_row(c, b, h, base + i);
    if (row < 0) {  // warp-uniform
      if (lane == 0) atomicOr(err, kFlagBadPage);
      continue;
    }
    const __half s = quantize_vals_warp<D>(x, (t ? c.v_codes : c.k_codes) + row * (D / 2),
                                           (t ? c.v_scales : c.k_scales) + row, lane);
    if (lane == 0) atomicMax(reinterpret_cast<int *>(&smax[ht]), __float_as_int(__half2float(s)));  // s >= 0
  }
  __syncthreads();
  for (int ht = threadIdx.x; ht < 2 * f.hkv; ht += blockDim.x) {
    const int h = ht >> 1, t = ht & 1;
    const int64_t bh = static_cast<int64_t>(b) * f.hkv + h;
    float *range = t ? f.v_range : f.k_range;
    const float r = fmaxf(range[bh], 7.f * smax[ht]);
    range[bh] = r;
    (t ? f.v_scale : f.k_scale)[bh] = __half_as_ushort(universal_scale(r));
  }
  if (threadIdx.x == 0) f.count[b] = 0;
}

}  // namespace

cudaError_t launch_flashq_init(const FlashqView &f, const KvView &c, const int32_t *cache_lens, int batch,
                               cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  flashq_init_kernel<<<batch * f.hkv * 2, 256, 0, stream>>>(f, c, cache_lens, batch);
  return cudaGetLastError();
}

cudaError_t launch_flashq_append(const void *k, const void *v, bool fp16_in, const FlashqView &f, int batch,
                                 uint32_t *err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const int threads = 32 * min(2 * f.hkv, 32);
  if (f.head_dim == 128) {
    if (fp16_in)
      flashq_append_kernel<__half, 128><<<batch, threads, 0, stream>>>(static_cast<const __half *>(k),
                                                                      static_cast<const __half *>(v), f, batch, err);
    else
      flashq_append_kernel<float, 128><<<batch, threads, 0, stream>>>(static_cast<const float *>(k),
                                                                     static_cast<const float *>(v), f, batch, err);
  } else {
    if (fp16_in)
      flashq_append_kernel<__half, 64><<<batch, threads, 0, stream>>>(static_cast<const __half *>(k),
                                                                     static_cast<const __half *>(v), f, batch, err);
    else
      flashq_append_kernel<float, 64><<<batch, threads, 0, stream>>>(static_cast<const float *>(k),
                                                                    static_cast<const float *>(v), f, batch, err);
  }
  return cudaGetLastError();
}

cudaError_t launch_flashq_attend(const uint16_t *q, const FlashqView &f, int batch, int hq, float scale_log2,
                                 uint16_t *out, float *lse, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const unsigned rows = static_cast<unsigned>(batch) * static_cast<unsigned>(hq);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return f.head_dim == 128 ? cudaLaunchKernelEx(&cfg, flashq_attend_kernel<128>, q, f, batch, hq, scale_log2, out, lse)
                           : cudaLaunchKernelEx(&cfg, flashq_attend_kernel<64>, q, f, batch, hq, scale_log2, out, lse);
}

cudaError_t launch_flashq_flush(const FlashqView &f, const KvView &c, const int32_t *cache_lens, int batch,
                                uint32_t *err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  if (f.head_dim == 128)
    flashq_flush_kernel<128><<<batch, 512, 0, stream>>>(f, c, cache_lens, batch, err);
  else
    flashq_flush_kernel<64><<<batch, 512, 0, stream>>>(f, c, cache_lens, batch, err);
  return cudaGetLastError();
}

}  // namespace qattn
