// Bounded mbarrier waits shared by the attention kernel and the library's
// wait self-test.  A wait that runs out records BSA_ERR_DEVICE_TIMEOUT in the
// caller's status word and in the CTA's abort flag and returns false; a CTA
// that sees another CTA's nonzero status stops at its next check.  No wait
// traps or spins without a limit.
#pragma once

#include <stdint.h>

#include "bsa.h"
#include "sm103_ptx.cuh"

namespace bsa {
namespace wait {

constexpr uint64_t kWaitTimeoutNs = 4000000000ull;   // 4 s: no legitimate wait comes close
constexpr uint64_t kDrainTimeoutNs = 200000000ull;   // 0.2 s per in-flight copy on abort

struct Ctl {
  volatile int *abort_flag;
  int32_t *dev_status;
};

__device__ __forceinline__ void report(const Ctl &c, int code) {
  *c.abort_flag = 1;
  if (c.dev_status != nullptr) atomicCAS(c.dev_status, 0, code);
}

// Bounded wait for phase `parity` of `bar`; false if this CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl &c,
                                         uint64_t limit_ns = kWaitTimeoutNs) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*c.abort_flag) return false;
      // another CTA already gave up: stop at once instead of waiting out our own limit
      if (c.dev_status != nullptr && *reinterpret_cast<volatile int32_t *>(c.dev_status) != 0) {
        *c.abort_flag = 1;
        return false;
      }
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        report(c, BSA_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// Wait that ignores the abort flag (used to drain in-flight work on abort).
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kDrainTimeoutNs) return;
  }
}

}  // namespace wait
}  // namespace bsa
