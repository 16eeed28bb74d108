// Kernel instances for state dtype f32 (p, m, v) and gradient dtype f32:
// every param-out dtype, and the param-remainder form.  One translation
// unit per (state, gradient) pair keeps the build parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry kernel_sf32_gf32(int out_dtype, bool remainders) {
  return kernel_for<FADAM_DT_F32, FADAM_DT_F32>(out_dtype, remainders);
}

}  // namespace fadam
