// Scalar backward kernels, fp32 gates and gradients.
#include "scan_scalar.cuh"

namespace scan {
cudaError_t launch_scalar_bwd_f32(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  return launch_scalar<LinOp, MODE_BWD, float>(p, pl, s);
}
}  // namespace scan
