// health.cu -- qattn_check_wait_timeout: a run-time check of the bounded
// mbarrier waits that every kernel of the library relies on to end instead of
// hanging when a pipeline partner never arrives.
//
// One warp initialises an mbarrier that expects one arrival, and thread 0
// waits for its first phase with the same bounded wait the attention kernels
// use.  Nothing ever arrives, so the wait must give up after `limit` cycles
// and record QATTN_FLAG_WAIT_TIMEOUT in the caller's word.
#include "../../include/qattn.h"
#include "internal.h"
#include "ptx.cuh"

namespace qattn {
namespace {

__global__ void wait_timeout_kernel(uint32_t *flags, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    *flags = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, flags, limit);
}

}  // namespace
}  // namespace qattn

extern "C" qattn_status qattn_check_wait_timeout(uint32_t *flags, int64_t limit_cycles, qattn_stream_t stream) {
  using namespace qattn;
  if (!flags || limit_cycles < 1 || limit_cycles > (int64_t(1) << 31)) {
    record_error("qattn_check_wait_timeout: flags must be a device pointer and 1 <= limit_cycles <= 2^31");
    return QATTN_ERR_INVALID_ARG;
  }
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(flags, static_cast<long long>(limit_cycles));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_error(cudaGetErrorString(e));
    return QATTN_ERR_CUDA;
  }
  return QATTN_OK;
}
