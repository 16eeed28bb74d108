// Kernel instances for an fp32 master with fp16 moments (m, v) and
// gradient dtype bf16: every param-out dtype.  One translation unit per
// (state form, gradient) pair keeps the build parallel.
#include "fadam_kernel.cuh"

namespace fadam {

KernelEntry kernel_sf32mf16_gbf16(int out_dtype, bool remainders) {
  return kernel_for<kStateF32MomF16, FADAM_DT_BF16>(out_dtype, remainders);
}

}  // namespace fadam
