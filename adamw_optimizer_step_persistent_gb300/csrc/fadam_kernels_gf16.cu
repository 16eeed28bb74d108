// Kernel instances for gradients of dtype f16 (every param-out dtype, and the
// param-remainder form).  One translation unit per gradient dtype keeps the
// build parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry kernel_gf16(int out_dtype, bool remainders) {
  return kernel_for<FADAM_DT_F16>(out_dtype, remainders);
}

}  // namespace fadam
