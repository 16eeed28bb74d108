// Plain kernel instances with reciprocal bias corrections
// (FADAM_RECIP_BC) for state dtype f16 and gradient dtype f16: every
// param-out dtype.  Apart from the default instances so that the build
// stays parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry recip_kernel_sf16_gf16(int out_dtype) {
  return recip_kernel_for<FADAM_DT_F16, FADAM_DT_F16, false>(out_dtype);
}

}  // namespace fadam
