// Kernel instances for gradients of dtype bf16 (every param-out dtype, and the
// param-remainder form).  One translation unit per gradient dtype keeps the
// build parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry kernel_gbf16(int out_dtype, bool remainders) {
  return kernel_for<FADAM_DT_BF16>(out_dtype, remainders);
}

}  // namespace fadam
