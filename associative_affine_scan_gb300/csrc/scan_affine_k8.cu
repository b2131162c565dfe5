// Block-matrix scan kernels for k = 8, every v in {1, 2, 4, 8, 16} (one
// translation unit per k so the builds run in parallel).
#include "scan_affine_generic.cuh"

namespace scan {

cudaError_t launch_affine_generic_k8(const AffineParams& p, int mode, cudaStream_t s) {
  return affg::launch_k<8>(p, mode, s);
}

}  // namespace scan
