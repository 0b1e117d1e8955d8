// e4m3 (fp8) input helpers shared by the kernels that read fp8 Q, K or V.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace bsa {

// Eight e4m3 values (low byte first) as floats, through the hardware's
// exact e4m3 -> f16 conversion.
__device__ __forceinline__ void e4m3x8_to_f32(const uint2 &u, float f[8]) {
  const uint32_t w[2] = {u.x, u.y};
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const __half2_raw hr =
          __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>((w[e] >> (16 * p)) & 0xFFFFu), __NV_E4M3);
      __half2 h;
      h = *reinterpret_cast<const __half2 *>(&hr);
      const float2 ff = __half22float2(h);
      f[4 * e + 2 * p] = ff.x;
      f[4 * e + 2 * p + 1] = ff.y;
    }
}

}  // namespace bsa
