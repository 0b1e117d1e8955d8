// bsa_select_mask_noalloc: the block-selection entry point for callers that
// cannot allocate device memory.
//
// bsa_select_mask needs a scratch buffer (the per-block mean queries and mean
// query norms, their tf32 splits and the two block-score matrices) that the
// caller allocates.  Some callers cannot do that: a host framework that owns
// the whole device memory pool and forbids allocations outside it, or a
// latency-critical caller that must not call cudaMalloc because it can
// synchronise the device.  This variant keeps its scratch in a fixed-size
// array that lives in the library's own device image, so the call itself
// allocates nothing.
//
// Costs and rules (also stated in include/bsa.h):
//   * every GPU that loads libbsa holds kScratchBytes of device memory for this
//     array until the process exits;
//   * shapes whose scratch exceeds kScratchBytes are rejected with
//     BSA_ERR_WORKSPACE before anything is launched;
//   * all calls on one device share the array, so calls whose kernels overlap
//     on the GPU (different streams without ordering) race and give wrong
//     results; calls ordered on one stream are fine.  Nothing in the array has
//     to start at zero: the pooling and scoring kernels overwrite every value
//     the selection reads, for both query aggregations;
//   * the first call on a device (and the first call after that device's
//     context was reset) looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

constexpr size_t kScratchBytes = 12u << 20;  // 12 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

// The address is cached per device together with the id of the context it was
// looked up in: a device reset creates a new primary context (with a new id)
// into which the module is loaded again, possibly at another address.
struct Cached {
  unsigned long long ctx_id;
  void *ptr;
};

std::mutex g_mutex;
Cached g_cache[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Unique id of the current context, or 0 if there is none or it cannot be read
// (the address is then looked up again, which is cheap once the module is loaded).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_select_scratch on the current device.
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  Cached &c = g_cache[dev];
  const unsigned long long id = current_context_id();
  // no current context yet (first use, or right after a reset): the lookup below makes the
  // device's primary context current
  if (c.ptr == nullptr || id == 0 || id != c.ctx_id) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    c.ptr = p;
    c.ctx_id = current_context_id();
  }
  *out = c.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" bsa_status bsa_select_mask_noalloc(const bsa_shape *shape, const bsa_select_params *params,
                                              const void *q, const float *centroid,
                                              const float *radius, const float *alpha,
                                              int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask,
                                              int32_t *dev_status, bsa_stream_t stream) {
  const size_t need = bsa_select_workspace_bytes(shape);  // 0 for an invalid shape
  if (need == 0)  // the regular entry point reports which shape check failed, before any launch
    return bsa_select_mask(shape, params, q, centroid, radius, alpha, kv_idx, kv_cnt, mask, nullptr,
                           0, dev_status, stream);
  if (need > kScratchBytes) return BSA_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return BSA_ERR_CUDA;
  // bsa_select_mask validates the parameters, flags (BSA_SELECT_TOKEN_MAX included) and
  // pointers exactly as for a caller-provided workspace, and forwards dev_status to the
  // score kernels, whose bounded waits report BSA_ERR_DEVICE_TIMEOUT there
  return bsa_select_mask(shape, params, q, centroid, radius, alpha, kv_idx, kv_cnt, mask, scratch,
                         kScratchBytes, dev_status, stream);
}
