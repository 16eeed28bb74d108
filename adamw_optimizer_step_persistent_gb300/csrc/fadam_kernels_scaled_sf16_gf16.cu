// Scaled-state kernel instances for state dtype f16 (p, m, v stored with
// one fp32 scale each per tensor) and gradient dtype f16: every param-out
// dtype.  Kept apart from the plain instances so the build stays parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry scaled_kernel_sf16_gf16(int out_dtype) {
  return scaled_kernel_for<FADAM_DT_F16, FADAM_DT_F16>(out_dtype);
}

}  // namespace fadam
