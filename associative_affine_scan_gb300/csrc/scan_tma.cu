// scan_tma.cu -- host side of the stream variant: tensor maps for 2-D tensor
// copies (TMA) of the flat [n / E, E] view of a scan tensor.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "scan_internal.h"

namespace scan {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// The encoder lives in the driver; the runtime hands out its entry point, so
// the library needs no link-time dependency on libcuda.
void load_encoder() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess && fn)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

bool encode_tile_map(CUtensorMap* m, const void* ptr, int elt, int64_t n, int J) {
  std::call_once(g_encode_once, load_encoder);
  if (!g_encode || !ptr || (elt != 2 && elt != 4) || (J != 1 && J != 2 && J != 4)) return false;
  if (reinterpret_cast<uintptr_t>(ptr) % 16) return false;
  const int E = tma_row_elems(elt);
  const int64_t rows = n / E;
  if (rows < 1 || rows > (1LL << 32)) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {(cuuint32_t)E, (cuuint32_t)(128 * J / E)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elt == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 128-byte rows of a flat buffer as a [rows, 32] fp32 tensor; the box is
// box_rows whole rows (at most 256), written to shared memory with the
// 128-byte swizzle.
bool encode_rows_map(CUtensorMap* m, const void* ptr, int64_t rows, int box_rows) {
  std::call_once(g_encode_once, load_encoder);
  if (!g_encode || !ptr || rows < 1 || rows > (1LL << 32) || box_rows < 1 || box_rows > 256)
    return false;
  if (reinterpret_cast<uintptr_t>(ptr) % 16) return false;
  const cuuint64_t dims[2] = {32, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A [B, T, N, 4, 4] fp32 tensor as {16 floats, N, T, B}: a box is 8 lanes x
// box_steps steps of one batch row, written to shared memory with the 64-byte
// swizzle (16-byte piece q of a 64-byte block lands at q ^ ((address >> 7) & 3)).
bool encode_blocks_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t N,
                       int box_steps) {
  std::call_once(g_encode_once, load_encoder);
  if (!g_encode || !ptr || B < 1 || T < 1 || N < 1 || box_steps < 1 || box_steps > 256) return false;
  if (reinterpret_cast<uintptr_t>(ptr) % 16) return false;
  if (N > (1LL << 32) || T > (1LL << 32) || B > (1LL << 32)) return false;
  const cuuint64_t dims[4] = {16, (cuuint64_t)N, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {64, (cuuint64_t)N * 64, (cuuint64_t)(N * T) * 64};
  const cuuint32_t box[4] = {16, 8, (cuuint32_t)box_steps, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(ptr), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace scan
