// Scaled-state kernel instances with reciprocal bias corrections
// (FADAM_RECIP_BC) for state dtype f16 and gradient dtype f32: every
// param-out dtype.  Apart from the default instances so that the build
// stays parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry recip_scaled_kernel_sf16_gf32(int out_dtype) {
  return recip_kernel_for<FADAM_DT_F16, FADAM_DT_F32, true>(out_dtype);
}

}  // namespace fadam
