// ptx.cuh -- thin inline-PTX wrappers used by the sm_103a kernels.
//
// Only public PTX ISA instructions are used (mbarrier, cp.async.bulk[.tensor],
// ldmatrix, movmatrix, mma.sync, griddepcontrol).  Every spin-wait is
// bounded: after kWaitCycles it sets a flag in the caller's status word and
// returns false instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qattn {

// Bits of the device status word (match QATTN_FLAG_* in qattn.h).
enum : uint32_t {
  kFlagWaitTimeout = 1u,  // an mbarrier wait gave up
  kFlagBadPage = 2u,      // a page id or length was out of range (rows skipped)
  kFlagTmem = 4u,         // tensor-memory allocation failed
};

// ~2 s at 2 GHz: far above any legitimate wait, far below a watchdog.
constexpr long long kWaitCycles = 4000000000LL;
// After a first timeout a kernel drains with waits this short (~1 ms).
constexpr long long kDrainCycles = 2000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t *err,
                                          long long limit = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      if (err) atomicOr(err, kFlagWaitTimeout);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------- bulk / TMA copies
// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled TMA load; c0 is the innermost coordinate (in elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                            int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// 3-D tiled TMA load; c0 is the innermost coordinate (in elements).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                            int32_t c1, int32_t c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------- programmatic launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------ thread-block cluster
// Cluster-wide barrier: every thread of the cluster that has not exited
// arrives (release) and waits for the others (acquire); executed by whole
// warps.  A hardware barrier, not a spin loop.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of `addr` (this CTA's shared memory) in the
// CTA of rank `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ------------------------------------------------------------- warp matrix
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// D = A(16x16, row) * B(16x8, col) + D, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// --------------------------------------------------------- nibble decoding
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t mask, uint32_t x) {
  // (a & mask) ^ x in one LOP3 (truth table 0x6a = (a & b) ^ c).
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(a), "r"(mask), "r"(x));
  return d;
}

// Decode the four nibble positions of each 16-bit half of `w` into exact
// fp16 integers.  A two's-complement nibble n holding code c satisfies
// n ^ 8 = c + 8, so placing (n ^ 8) in the mantissa of 1024.0 gives
// 1032 + c (nibble in bits 0-3) or 1024 + 16 (c + 8) (bits 4-7); one fp16
// subtract or fma then yields c exactly.
//   out[k] = (code at nibble k of the low half, code at nibble k of the high half)
__device__ __forceinline__ void decode_nibbles(uint32_t w, uint32_t (&out)[4]) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 kSixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
  const __half2 kMinus72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
  const uint32_t w8 = w >> 8;
  uint32_t x0 = lop3_and_xor(w, 0x000F000Fu, 0x64086408u);
  uint32_t x1 = lop3_and_xor(w, 0x00F000F0u, 0x64806480u);
  uint32_t x2 = lop3_and_xor(w8, 0x000F000Fu, 0x64086408u);
  uint32_t x3 = lop3_and_xor(w8, 0x00F000F0u, 0x64806480u);
  __half2 h0 = __hsub2(*reinterpret_cast<__half2 *>(&x0), k1032);
  __half2 h1 = __hfma2(*reinterpret_cast<__half2 *>(&x1), kSixteenth, kMinus72);
  __half2 h2 = __hsub2(*reinterpret_cast<__half2 *>(&x2), k1032);
  __half2 h3 = __hfma2(*reinterpret_cast<__half2 *>(&x3), kSixteenth, kMinus72);
  out[0] = *reinterpret_cast<uint32_t *>(&h0);
  out[1] = *reinterpret_cast<uint32_t *>(&h1);
  out[2] = *reinterpret_cast<uint32_t *>(&h2);
  out[3] = *reinterpret_cast<uint32_t *>(&h3);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// 2^x (hardware approximation, flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset inside a 1024-byte-aligned tile written by TMA with
// CU_TENSOR_MAP_SWIZZLE_128B: the 16-byte chunk index (bits 4-6) is XORed
// with the 128-byte row index modulo 8 (bits 7-9).
__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }

}  // namespace qattn
