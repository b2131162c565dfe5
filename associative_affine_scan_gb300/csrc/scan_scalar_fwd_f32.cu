// Scalar forward kernels, fp32 inputs.
#include "scan_scalar.cuh"

namespace scan {
cudaError_t launch_scalar_fwd_f32(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  return launch_scalar<LinOp, MODE_FWD, float>(p, pl, s);
}
}  // namespace scan
