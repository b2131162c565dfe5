// Scalar backward kernels, bf16 gates and gradients (fp32 accumulation).
#include "scan_scalar.cuh"

namespace scan {
cudaError_t launch_scalar_bwd_bf16(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  return launch_scalar<LinOp, MODE_BWD, __nv_bfloat16>(p, pl, s);
}
}  // namespace scan
