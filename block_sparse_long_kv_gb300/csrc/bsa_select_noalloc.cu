// bsa_select_mask_noalloc: the block-selection entry point for callers that
// cannot allocate device memory.
//
// bsa_select_mask needs a scratch buffer (the per-block mean queries and mean
// query norms) that the caller allocates.  Some callers cannot do that: a host
// framework that owns the whole device memory pool and forbids allocations
// outside it, or a latency-critical caller that must not call cudaMalloc
// because it can synchronise the device.  This variant keeps its scratch in a
// fixed-size array that lives in the library's own device image, so the call
// itself allocates nothing.
//
// Costs and rules (also stated in include/bsa.h):
//   * every GPU that loads libbsa holds kScratchBytes of device memory for this
//     array until the process exits;
//   * shapes whose scratch exceeds kScratchBytes are rejected with
//     BSA_ERR_WORKSPACE;
//   * all calls on one device share the array, so calls whose kernels overlap
//     on the GPU (different streams without ordering) race and give wrong
//     results; calls ordered on one stream are fine.  Nothing in the array has
//     to start at zero: the query-pooling kernel overwrites every value the
//     scoring kernel reads;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

constexpr size_t kScratchBytes = 12u << 20;  // 12 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_select_scratch on the current device (looked up once).
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" bsa_status bsa_select_mask_noalloc(const bsa_shape *shape, const bsa_select_params *params,
                                              const void *q, const float *centroid,
                                              const float *radius, const float *alpha,
                                              int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask,
                                              int32_t *dev_status, bsa_stream_t stream) {
  (void)dev_status;  // the select kernels have no waits
  const size_t need = bsa_select_workspace_bytes(shape);  // 0 for an invalid shape
  if (need == 0)  // the regular entry point reports which shape check failed, before any launch
    return bsa_select_mask(shape, params, q, centroid, radius, alpha, kv_idx, kv_cnt, mask, nullptr,
                           0, dev_status, stream);
  if (need > kScratchBytes) return BSA_ERR_WORKSPACE;
  if (!params || !q || !centroid || !radius || !alpha || !kv_idx || !kv_cnt)
    return BSA_ERR_INVALID_ARG;
  if (!(params->centroid_keep >= 0.f && params->centroid_keep <= 1.f) ||
      !(params->rescue_keep >= 0.f && params->rescue_keep <= 1.f) || params->flags != 0)
    return BSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(centroid) || !aligned16(radius) || !aligned16(alpha) ||
      !aligned16(kv_idx) || !aligned16(kv_cnt) || (mask && !aligned16(mask)))
    return BSA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return BSA_ERR_CUDA;
  return bsa_select_mask(shape, params, q, centroid, radius, alpha, kv_idx, kv_cnt, mask, scratch,
                         kScratchBytes, dev_status, stream);
}
