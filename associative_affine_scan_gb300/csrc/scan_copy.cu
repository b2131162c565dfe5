// scan_copy.cu -- scan_copy: the device-to-device copies that give the
// achievable-bandwidth ceiling the scan kernels are measured against.
//
// A scan moves every element through HBM once in each direction it needs
// (12 bytes per element forward, 20 backward), so the ceiling it can reach is
// that of a plain read + write stream on the same GPU. Two hand-written
// copies, launched the way the scan kernels are (on the caller's stream, one
// wave of blocks sized from the SM count):
//   - SCAN_COPY_VEC: every thread moves 4 x 16 bytes per trip with streaming
//     128-bit loads and stores, grid-stride over the buffer (the access the
//     register-path scan kernels use);
//   - SCAN_COPY_TMA: one thread per block moves 32 KB tiles (256 rows of 128
//     bytes) through a 3-stage shared-memory ring with 2-D tensor copies: a
//     tile load completes on its stage's mbarrier, the tile is stored back
//     with a tensor store, and the stage is refilled once that store has
//     read it (the copy path of the scan's stream variant).
// Every mbarrier wait is bounded; on expiry the kernel sets the caller's
// status word to SCAN_ERR_TIMEOUT, waits (bounded) for its loads in flight and
// its stores, and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/libscan.h"
#include "scan_internal.h"
#include "scan_scalar.cuh"

namespace {

using namespace scan;

constexpr int kVecThreads = 256;
constexpr int kVecUnroll = 4;
constexpr int kTileRows = 256;                   // rows of 128 bytes per tile
constexpr unsigned kTileBytes = kTileRows * 128;  // 32 KB
constexpr int kCopyStages = 3;
constexpr int kTmaBlocksPerSm = 2;
constexpr unsigned long long kCopyWaitNs = 1000000000ULL;

__global__ void __launch_bounds__(kVecThreads) copy_vec_kernel(const uint4* __restrict__ src,
                                                               uint4* __restrict__ dst,
                                                               int64_t n16) {
  const int64_t step = (int64_t)gridDim.x * kVecThreads * kVecUnroll;
  for (int64_t base = (int64_t)blockIdx.x * kVecThreads * kVecUnroll + threadIdx.x; base < n16;
       base += step) {
    uint4 v[kVecUnroll];
#pragma unroll
    for (int u = 0; u < kVecUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kVecThreads;
      if (i < n16) v[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kVecUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kVecThreads;
      if (i < n16) __stcs(dst + i, v[u]);
    }
  }
}

__global__ void __launch_bounds__(32) copy_tma_kernel(const __grid_constant__ CUtensorMap src,
                                                      const __grid_constant__ CUtensorMap dst,
                                                      int64_t tiles, unsigned* status) {
  extern __shared__ __align__(1024) unsigned char copy_smem[];
  __shared__ unsigned long long bars[kCopyStages];
  if (threadIdx.x != 0) return;
  // the 128-byte swizzle wants 1024-byte aligned tiles
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(copy_smem) + 1023) & ~static_cast<uintptr_t>(1023));
  for (int s = 0; s < kCopyStages; ++s) mbar_init(&bars[s], 1);
  fence_mbar_init();
  const int64_t first = blockIdx.x;
  const int64_t count = tiles > first ? (tiles - 1 - first) / gridDim.x + 1 : 0;
  auto row_of = [&](int64_t i) { return (int)((first + i * (int64_t)gridDim.x) * kTileRows); };
  auto issue = [&](int64_t i) {
    const int s = (int)(i % kCopyStages);
    mbar_expect_tx(&bars[s], kTileBytes);
    tma_load_2d(ring + (size_t)s * kTileBytes, &src, 0, row_of(i), &bars[s]);
  };
  const int64_t pre = count < kCopyStages - 1 ? count : kCopyStages - 1;
  for (int64_t i = 0; i < pre; ++i) issue(i);
  int64_t i = 0;
  for (; i < count; ++i) {
    const int s = (int)(i % kCopyStages);
    if (!mbar_wait(&bars[s], (unsigned)((i / kCopyStages) & 1), kCopyWaitNs)) break;
    tma_store_2d(&dst, 0, row_of(i), ring + (size_t)s * kTileBytes);
    bulk_commit();
    const int64_t j = i + kCopyStages - 1;
    if (j < count) {
      bulk_wait_read<1>();  // the store of tile i - 1 has read stage j % kCopyStages
      issue(j);
    }
  }
  if (i < count) {
    if (status) atomicExch(status, (unsigned)SCAN_ERR_TIMEOUT);
    const int64_t issued = i + kCopyStages - 1 < count ? i + kCopyStages - 1 : count;
    for (int64_t k = i; k < issued; ++k)
      (void)mbar_wait(&bars[k % kCopyStages], (unsigned)((k / kCopyStages) & 1), kCopyWaitNs);
  }
  bulk_wait_all();
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

extern "C" scan_status scan_copy(const void* src, void* dst, size_t bytes, int32_t mode,
                                 uint32_t* status, cudaStream_t stream) {
  if (mode != SCAN_COPY_VEC && mode != SCAN_COPY_TMA) return SCAN_ERR_INVALID_ARG;
  if (bytes == 0) return SCAN_OK;
  if (!src || !dst) return SCAN_ERR_INVALID_ARG;
  if ((uintptr_t)src % 16 || (uintptr_t)dst % 16) return SCAN_ERR_ALIGNMENT;
  const int sms = sm_count();
  if (sms <= 0) return SCAN_ERR_CUDA;
  if (mode == SCAN_COPY_VEC) {
    if (bytes % 16) return SCAN_ERR_INVALID_ARG;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, copy_vec_kernel, kVecThreads, 0) !=
            cudaSuccess ||
        per_sm <= 0)
      return SCAN_ERR_CUDA;
    const int64_t n16 = (int64_t)(bytes / 16);
    const int64_t need = (n16 + kVecThreads * kVecUnroll - 1) / (kVecThreads * kVecUnroll);
    const int64_t wave = (int64_t)sms * per_sm;
    const int grid = (int)(need < wave ? need : wave);
    copy_vec_kernel<<<grid, kVecThreads, 0, stream>>>(static_cast<const uint4*>(src),
                                                      static_cast<uint4*>(dst), n16);
    return cudaGetLastError() == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
  }
  if (bytes % 128) return SCAN_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)(bytes / 128);
  if (rows > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;  // row coordinates are int32
  CUtensorMap ms, md;
  if (!encode_rows_map(&ms, src, rows, kTileRows) || !encode_rows_map(&md, dst, rows, kTileRows))
    return SCAN_ERR_CUDA;
  const size_t smem = (size_t)kCopyStages * kTileBytes + 1024;
  if (cudaFuncSetAttribute(copy_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SCAN_ERR_CUDA;
  const int64_t tiles = (rows + kTileRows - 1) / kTileRows;
  const int64_t wave = (int64_t)sms * kTmaBlocksPerSm;
  const int grid = (int)(tiles < wave ? tiles : wave);
  copy_tma_kernel<<<grid, 32, smem, stream>>>(ms, md, tiles, status);
  return cudaGetLastError() == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}
