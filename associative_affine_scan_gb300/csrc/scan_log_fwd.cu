// Log-space forward kernels (fp32).
#include "scan_scalar.cuh"

namespace scan {
cudaError_t launch_log_fwd(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  return launch_scalar<LogOp, MODE_FWD, float>(p, pl, s);
}
}  // namespace scan
