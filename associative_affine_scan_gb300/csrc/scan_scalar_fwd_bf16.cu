// Scalar forward kernels, bf16 inputs (fp32 accumulation and output).
#include "scan_scalar.cuh"

namespace scan {
cudaError_t launch_scalar_fwd_bf16(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  return launch_scalar<LinOp, MODE_FWD, __nv_bfloat16>(p, pl, s);
}
}  // namespace scan
