// Log-space backward kernels (fp32): the linear adjoint on exp(log a).
#include "scan_scalar.cuh"

namespace scan {
cudaError_t launch_log_bwd(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  return launch_scalar<LinOp, MODE_LOGBWD, float>(p, pl, s);
}
}  // namespace scan
