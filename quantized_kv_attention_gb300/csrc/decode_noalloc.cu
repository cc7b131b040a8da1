// decode_noalloc.cu -- qattn_decode_noalloc: split-KV decode for callers that
// cannot allocate device memory.
//
// qattn_decode needs a caller-provided workspace for its split partials.  Some
// callers have no way to get one: a plugin loaded into an inference engine
// that only hands it input and output buffers, code running on a device
// whose memory a caching allocator reserved up front, or a latency-critical
// loop that must not call cudaMalloc (which can synchronize the device).
// This entry point gives them the same kernels with the partials in a fixed
// array that the library owns: QATTN_NOALLOC_SCRATCH_BYTES of device memory
// on every GPU that loads the library, held until the process exits.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress; make that first call
// before any stream capture.  Every call on a device shares the one array, so
// calls that overlap on the GPU (different streams, no ordering) race.  No
// part of the array has to start at zero: each call writes every partial
// value and lse it later reads.  Nothing here allocates.
#include <stdio.h>

#include <mutex>

#include "../../include/qattn.h"
#include "internal.h"

namespace qattn {
namespace {

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a device address; kernels get the address from set-up.
static __device__ __align__(256) unsigned char g_decode_scratch[QATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;

struct ScratchSlot {
  std::once_flag once;
  void *ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchSlot g_slots[kMaxScratchDevices];

}  // namespace
}  // namespace qattn

extern "C" qattn_status qattn_decode_noalloc(const uint16_t *q, const qattn_kv_cache *cache,
                                             const int32_t *seq_lens, int32_t batch,
                                             int32_t num_q_heads, int32_t max_seq_len,
                                             float softmax_scale, int32_t num_splits,
                                             uint16_t *out, float *lse, qattn_stream_t stream) {
  using namespace qattn;
  char msg[256];
  // Size first: a request whose partials do not fit is refused before any
  // device work (qattn_decode validates everything else).
  // a listed cache's split rows follow the model's group size
  const int32_t ws_hkv = cache ? (cache->kv_head_index ? cache->model_kv_heads : cache->num_kv_heads) : 0;
  const size_t need = qattn_decode_workspace_size(batch, num_q_heads, ws_hkv, cache ? cache->head_dim : 0,
                                                  max_seq_len, num_splits);
  if (need > QATTN_NOALLOC_SCRATCH_BYTES) {
    snprintf(msg, sizeof(msg),
             "qattn_decode_noalloc: these sizes need %zu bytes of split scratch, more than the "
             "%u-byte static scratch; use fewer splits or qattn_decode with a workspace",
             need, (unsigned)QATTN_NOALLOC_SCRATCH_BYTES);
    record_error(msg);
    return QATTN_ERR_UNSUPPORTED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    snprintf(msg, sizeof(msg), "qattn_decode_noalloc: no usable current device (%s)",
             e != cudaSuccess ? cudaGetErrorString(e) : "device index out of range");
    record_error(msg);
    return e != cudaSuccess ? QATTN_ERR_CUDA : QATTN_ERR_UNSUPPORTED;
  }
  ScratchSlot &slot = g_slots[dev];
  std::call_once(slot.once, [&slot]() {
    slot.err = cudaGetSymbolAddress(&slot.ptr, g_decode_scratch);
  });
  if (slot.err != cudaSuccess || slot.ptr == nullptr) {
    snprintf(msg, sizeof(msg), "qattn_decode_noalloc: cudaGetSymbolAddress of the scratch failed: %s",
             cudaGetErrorString(slot.err));
    record_error(msg);
    return QATTN_ERR_CUDA;
  }
  return qattn_decode(q, cache, seq_lens, batch, num_q_heads, max_seq_len, softmax_scale, num_splits,
                      slot.ptr, QATTN_NOALLOC_SCRATCH_BYTES, out, lse, stream);
}
