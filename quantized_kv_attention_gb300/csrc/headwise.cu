// headwise.cu -- the headwise mixed-precision plan (TurboAttention, arXiv
// 2412.08585, §3.2): a priority per kv-head from a prompt's keys and values,
// and the choice of the n_h lowest-priority heads for 2-bit storage.
//
// Per head and tensor, over the rows of every sequence (t < lens[b]):
//   mx_j, mn_j = largest and smallest value of channel j
//   gap_j = mx_j - mn_j,  gap = max_j mx_j - min_j mn_j
//   std   = sqrt(sum_j (gap_j - mean)^2 / D),  mean = sum_j gap_j / D
//   priority = gap * std   (the page names both statistics; their product is
//   this library's reading of the missing equation)
// A kv-head's priority is the larger of its key and value priorities; the
// n_h heads of lowest priority (ties: lower index first) get 2 bits.
//
// Three launches: clear the per-channel extrema, reduce the rows (one CTA per
// 256 rows of one (tensor, sequence, head), combined by atomic max / min on
// order-preserving integer keys), then one thread per head computes the
// statistics in binary64, in channel order, without fused multiply-adds (so
// the priorities, and hence the ranking, are reproducible bit for bit), and
// ranks the heads.
#include "internal.h"
#include "ptx.cuh"

namespace qattn {
namespace {

// Largest kv-head count of a plan; extrema of both tensors for every
// (head, channel): 2 * kMaxHeads * 128 keys each for max and min.
constexpr int kMaxHeads = 256;
__device__ uint32_t g_ext_max[2 * kMaxHeads * 128];
__device__ uint32_t g_ext_min[2 * kMaxHeads * 128];

// Order-preserving map of a finite float to an unsigned key.
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fval(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__global__ void __launch_bounds__(256) plan_clear_kernel(int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    g_ext_max[i] = 0u;           // below every key
    g_ext_min[i] = 0xffffffffu;  // above every key
  }
}

constexpr int kRowsPerCta = 256;

// grid (row chunks * batch * Hkv, 2 tensors); thread j % D reads channel j
// of rows j / D, j / D + 256 / D, ...
template <typename T, int D>
__global__ void __launch_bounds__(256)
    plan_reduce_kernel(const T *__restrict__ k, const T *__restrict__ v, int hkv, int n, int chunks,
                       const int32_t *__restrict__ lens) {
  constexpr int kPar = 256 / D;  // rows read in parallel
  const int64_t bh = blockIdx.x / chunks;
  const int b = static_cast<int>(bh / hkv), h = static_cast<int>(bh % hkv), tensor = blockIdx.y;
  int len = lens ? __ldg(lens + b) : n;
  len = len < 0 ? 0 : (len > n ? n : len);
  const int r0 = static_cast<int>(blockIdx.x % chunks) * kRowsPerCta;
  if (r0 >= len) return;
  const int r1 = min(len, r0 + kRowsPerCta);
  const T *src = (tensor ? v : k) + static_cast<int64_t>(bh) * n * D;
  const int j = threadIdx.x % D, rp = threadIdx.x / D;
  float mx = -INFINITY, mn = INFINITY;
  for (int r = r0 + rp; r < r1; r += kPar) {
    const float x = static_cast<float>(src[static_cast<int64_t>(r) * D + j]);
    mx = fmaxf(mx, x);
    mn = fminf(mn, x);
  }
  __shared__ float smx[256], smn[256];
  smx[threadIdx.x] = mx, smn[threadIdx.x] = mn;
  __syncthreads();
  if (rp == 0) {
#pragma unroll
    for (int p = 1; p < kPar; ++p) mx = fmaxf(mx, smx[p * D + j]), mn = fminf(mn, smn[p * D + j]);
    const int slot = (tensor * kMaxHeads + h) * D + j;
    atomicMax(g_ext_max + slot, fkey(mx));
    atomicMin(g_ext_min + slot, fkey(mn));
  }
}

// gap * std of one head and tensor from its extrema (binary64, channel order).
template <int D>
__device__ double tensor_priority(int tensor, int h) {
  const uint32_t *kmx = g_ext_max + (tensor * kMaxHeads + h) * D;
  const uint32_t *kmn = g_ext_min + (tensor * kMaxHeads + h) * D;
  double total = 0.0, top = -INFINITY, bottom = INFINITY;
  for (int j = 0; j < D; ++j) {
    const double a = fval(kmx[j]), z = fval(kmn[j]);
    total = __dadd_rn(total, __dsub_rn(a, z));
    top = fmax(top, a);
    bottom = fmin(bottom, z);
  }
  const double mean = __ddiv_rn(total, static_cast<double>(D));
  double sq = 0.0;
  for (int j = 0; j < D; ++j) {
    const double e = __dsub_rn(__dsub_rn(fval(kmx[j]), fval(kmn[j])), mean);
    sq = __dadd_rn(sq, __dmul_rn(e, e));
  }
  const double sd = __dsqrt_rn(__ddiv_rn(sq, static_cast<double>(D)));
  return __dmul_rn(__dsub_rn(top, bottom), sd);
}

// One CTA: thread h computes head h's priority, then every head counts the
// heads ranked before it.
template <int D>
__global__ void __launch_bounds__(kMaxHeads)
    plan_finish_kernel(int batch, int hkv, int n, const int32_t *__restrict__ lens, int n_low,
                       int32_t *__restrict__ bits, double *__restrict__ priority) {
  __shared__ double pr[kMaxHeads];
  __shared__ int any_rows;
  if (threadIdx.x == 0) {
    int rows = 0;
    for (int b = 0; b < batch && !rows; ++b) {
      const int len = lens ? __ldg(lens + b) : n;
      rows = min(len, n) > 0;
    }
    any_rows = rows;
  }
  __syncthreads();
  const int h = threadIdx.x;
  if (h < hkv) {
    const double p = any_rows ? fmax(tensor_priority<D>(0, h), tensor_priority<D>(1, h)) : 0.0;
    pr[h] = p;
    if (priority) priority[h] = p;
  }
  __syncthreads();
  if (h < hkv) {
    int rank = 0;
    for (int o = 0; o < hkv; ++o) rank += pr[o] < pr[h] || (pr[o] == pr[h] && o < h);
    bits[h] = rank < n_low ? 2 : 4;
  }
}

template <typename T, int D>
cudaError_t launch_p(const void *k, const void *v, int batch, int hkv, int n, const int32_t *lens, int n_low,
                     int32_t *bits, double *priority, cudaStream_t stream) {
  plan_clear_kernel<<<32, 256, 0, stream>>>(2 * kMaxHeads * D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (n > 0) {
    const int chunks = (n + kRowsPerCta - 1) / kRowsPerCta;
    dim3 grid(static_cast<unsigned>(static_cast<int64_t>(chunks) * batch * hkv), 2);
    plan_reduce_kernel<T, D><<<grid, 256, 0, stream>>>(static_cast<const T *>(k), static_cast<const T *>(v), hkv,
                                                      n, chunks, lens);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  plan_finish_kernel<D><<<1, kMaxHeads, 0, stream>>>(batch, hkv, n, lens, n_low, bits, priority);
  return cudaGetLastError();
}

}  // namespace

int headwise_max_heads() { return kMaxHeads; }

cudaError_t launch_headwise_plan(const void *k, const void *v, bool fp16_in, int batch, int hkv, int n,
                                 int head_dim, const int32_t *lens, int n_low, int32_t *bits, double *priority,
                                 cudaStream_t stream) {
  if (head_dim == 128)
    return fp16_in ? launch_p<__half, 128>(k, v, batch, hkv, n, lens, n_low, bits, priority, stream)
                   : launch_p<float, 128>(k, v, batch, hkv, n, lens, n_low, bits, priority, stream);
  return fp16_in ? launch_p<__half, 64>(k, v, batch, hkv, n, lens, n_low, bits, priority, stream)
                 : launch_p<float, 64>(k, v, batch, hkv, n, lens, n_low, bits, priority, stream);
}

}  // namespace qattn
