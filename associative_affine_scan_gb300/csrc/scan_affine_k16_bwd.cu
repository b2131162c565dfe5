// Block-matrix scan kernels for k = 16, every v in {1, 2, 4, 8, 16},
// backward only (the k = 16 instantiations are the slowest to
// compile, so each mode has its own translation unit).
#include "scan_affine_generic.cuh"

namespace scan {

cudaError_t launch_affine_generic_k16_bwd(const AffineParams& p, cudaStream_t s) {
  return affg::launch_k<16, MODE_BWD>(p, s);
}

}  // namespace scan
