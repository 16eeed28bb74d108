// Kernel instances for state dtype f32 (p, m, v) and gradient dtype bf16:
// every param-out dtype, and the param-remainder form.  One translation
// unit per (state, gradient) pair keeps the build parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry kernel_sf32_gbf16(int out_dtype, bool remainders) {
  return kernel_for<FADAM_DT_F32, FADAM_DT_BF16>(out_dtype, remainders);
}

}  // namespace fadam
