// combine.cu -- log-sum-exp merge of split-KV partials.
//
// The split-KV form of FlashAttention's online softmax (TurboAttention,
// arXiv 2412.08585, §2.2): each split c of the keys yields its output O_c
// normalised over that split and lse_c = ln sum_j exp(s_j); the exact result
// is O = sum_c exp(lse_c - L) O_c with L = ln sum_c exp(lse_c).  It is the
// single-GPU counterpart of the sequence-parallel attention the same section
// mentions (Ring / Striped / Lean attention).
//
// One CTA of 8 warps per output row: weights computed once into shared
// memory, then warp w accumulates splits w, w+8, ... with each lane owning
// D/32 consecutive outputs (coalesced fp32 loads), then a shared-memory sum.
#include <math.h>

#include "../../include/qattn.h"
#include "internal.h"
#include "ptx.cuh"

namespace qattn {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float block_reduce(float v, float *red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  __syncthreads();  // red is reused between calls
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    combine_kernel(const float *__restrict__ po, const float *__restrict__ pl, int splits,
                   int64_t rows, uint16_t *__restrict__ out, float *__restrict__ lse) {
  pdl_wait();  // partials come from the preceding kernel on the stream
  pdl_launch_dependents();  // before its own wait a dependent reads only sequence lengths (not written here)
  constexpr int VPL = D / 32;
  __shared__ float w[QATTN_MAX_SPLITS];
  __shared__ float red[kWarps];
  __shared__ float acc_s[kWarps][D];
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  float mx = -INFINITY;
  for (int s = tid; s < splits; s += kWarps * 32) mx = fmaxf(mx, pl[s * rows + row]);
  const float M = block_reduce(mx, red, true);
  if (M == -INFINITY) {  // no split saw a key
    for (int d = tid; d < D; d += kWarps * 32) out[row * D + d] = 0;
    if (tid == 0 && lse) lse[row] = -INFINITY;
    return;
  }
  float z = 0.f;
  for (int s = tid; s < splits; s += kWarps * 32) {
    const float l = pl[s * rows + row];
    const float e = l == -INFINITY ? 0.f : expf(l - M);
    w[s] = e;
    z += e;
  }
  const float Z = block_reduce(z, red, false);  // also orders the w[] writes

  float acc[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) acc[j] = 0.f;
#pragma unroll 4
  for (int s = warp; s < splits; s += kWarps) {
    const float ws = w[s];
    if (ws > 0.f) {  // empty splits are never read
      const float *src = po + (s * rows + row) * D + lane * VPL;
      if constexpr (VPL == 4) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(src));
        acc[0] += ws * x.x, acc[1] += ws * x.y, acc[2] += ws * x.z, acc[3] += ws * x.w;
      } else {
        const float2 x = __ldg(reinterpret_cast<const float2 *>(src));
        acc[0] += ws * x.x, acc[1] += ws * x.y;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j) acc_s[warp][lane * VPL + j] = acc[j];
  __syncthreads();
  const float inv = 1.f / Z;
  for (int d = tid; d < D; d += kWarps * 32) {
    float o = 0.f;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) o += acc_s[ww][d];
    out[row * D + d] = __half_as_ushort(__float2half_rn(o * inv));
  }
  if (tid == 0 && lse) lse[row] = M + logf(Z);
}

template <int D>
cudaError_t launch_c(const float *po, const float *pl, int splits, int64_t rows, uint16_t *out,
                     float *lse, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel<D>, po, pl, splits, rows, out, lse);
}

}  // namespace

cudaError_t launch_combine(const float *partial_o, const float *partial_lse, int splits,
                           int64_t rows, int head_dim, uint16_t *out, float *lse, bool pdl,
                           cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  return head_dim == 128 ? launch_c<128>(partial_o, partial_lse, splits, rows, out, lse, pdl, stream)
                         : launch_c<64>(partial_o, partial_lse, splits, rows, out, lse, pdl, stream);
}

}  // namespace qattn
