// Kernel instances for gradients of dtype f32 (every param-out dtype, and the
// param-remainder form).  One translation unit per gradient dtype keeps the
// build parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry kernel_gf32(int out_dtype, bool remainders) {
  return kernel_for<FADAM_DT_F32>(out_dtype, remainders);
}

}  // namespace fadam
