// Self-test of the device wait limits, with no compute: every CTA's first
// thread waits, through the same bounded wait the attention kernel uses, on an
// mbarrier that nothing completes.  CTA 0 gives up after the caller's limit and
// records BSA_ERR_DEVICE_TIMEOUT; the other CTAs wait with the library's own
// limit and must stop once they see that status.  The kernel always returns;
// nothing traps.

#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa.h"
#include "bsa_wait.cuh"

namespace bsa {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t *dev_status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const wait::Ctl ctl{&abort_flag, dev_status};
    wait::wait_bar(ptx::smem_addr(&bar), 0, ctl, blockIdx.x == 0 ? limit_ns : wait::kWaitTimeoutNs);
  }
}

}  // namespace
}  // namespace bsa

extern "C" bsa_status bsa_selftest_wait_timeout(int32_t *dev_status, uint64_t limit_ns, int32_t ctas,
                                                bsa_stream_t stream) {
  if (dev_status == nullptr || (reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0) return BSA_ERR_INVALID_ARG;
  if (limit_ns < 1000000ull || limit_ns > 1000000000ull || ctas < 1 || ctas > 8) return BSA_ERR_INVALID_ARG;
  bsa::wait_selftest_kernel<<<ctas, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      dev_status, static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}
