// Kernel instances for state dtype f16 (p, m, v) and gradient dtype f16:
// every param-out dtype.  One translation
// unit per (state, gradient) pair keeps the build parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry kernel_sf16_gf16(int out_dtype, bool remainders) {
  return kernel_for<FADAM_DT_F16, FADAM_DT_F16>(out_dtype, remainders);
}

}  // namespace fadam
