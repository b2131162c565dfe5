// scan_noalloc.cu -- scan_fwd_noalloc: the scalar forward scan for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// running inside a memory-capped or pre-partitioned arena, a real-time path
// that forbids allocation after start-up, or a plugin host that only passes
// in the tensors it owns. For them this entry point runs the look-back
// forward kernel (the one kernel here whose chunks need scratch memory for
// their published summaries) with its scratch in a fixed array that lives in
// the library itself.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/libscan.h"
#include "scan_internal.h"

namespace {

using namespace scan;

// The library's own scratch: header + one 16-byte summary record per
// (row, chunk). Every GPU that loads the library holds these bytes until the
// process exits. Static device memory starts zeroed.
constexpr size_t kScratchBytes = SCAN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device. In host code the
// symbol's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, called once per device with that device current.
// Nothing is written here: a __device__ array without an initialiser is
// zero-filled when the module is loaded, so the header (tile ticket, epoch,
// completion counter, status word) starts at 0 with no copy or memset that
// could race with a kernel already queued on another stream.
scan_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SCAN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SCAN_ERR_UNSUPPORTED;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SCAN_ERR_CUDA;
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return SCAN_OK;
}

// The scratch is per device and the launch goes to the current device: the
// tensors must live there (a pointer of another device is refused).
bool on_current_device(const void* ptr) {
  int dev = 0;
  cudaPointerAttributes at;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged
             ? at.device == dev
             : false;
}

}  // namespace

extern "C" scan_status scan_fwd_noalloc(const void* a, const void* x, const float* h0,
                                        const int32_t* cu_seqlens, int32_t n_seqs, float* h,
                                        int64_t B, int64_t C, int64_t T, scan_dtype dt,
                                        int32_t reverse, cudaStream_t stream) {
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  if (B < 0 || C < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (cu_seqlens && (B != 1 || n_seqs < 1 || T > 0x7fffffffLL)) return SCAN_ERR_INVALID_ARG;
  const int64_t rows = B * C;
  if (rows * T == 0) return SCAN_OK;
  if (!a || !x || !h) return SCAN_ERR_INVALID_ARG;

  // the same tiling as the workspace-based look-back: rows of 4, chunks of
  // 128, 256 or 512 steps, each row cut so 4-step groups are 16-byte aligned
  const int J = T <= 128 ? 1 : (T <= 256 ? 2 : 4);
  const int R = rows < 4 ? (int)rows : 4;
  const int64_t L = 128LL * J;
  const int64_t M = (T + ((T % 4) ? 3 : 0) + L - 1) / L;
  const int64_t G = (rows + R - 1) / R;
  const int64_t tiles = M * G;
  if (tiles > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;
  const size_t need = kWsHeaderBytes + (size_t)(rows * M) * 16u;
  if (need > kScratchBytes) return SCAN_ERR_WORKSPACE;  // beyond the fixed scratch

  if (!on_current_device(a) || !on_current_device(x) || !on_current_device(h))
    return SCAN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  scan_status st = scratch_on_current_device(&scratch);
  if (st != SCAN_OK) return st;

  auto aligned = [](const void* p, size_t n) { return ((uintptr_t)p % n) == 0; };
  const size_t va = dt == SCAN_BF16 ? 8 : 16;
  ScalarPlan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.variant = VAR_LOOKBACK;
  pl.J = J;
  pl.R = R;
  pl.M = (int)M;
  pl.G = (int)G;
  pl.vec = aligned(a, va) && aligned(x, va) && aligned(h, 16);
  pl.nseg = 1;
  pl.cps = (int)M;
  pl.ws_bytes = need;
  // as for scan_fwd: offsets staged in shared memory only when they all fit
  pl.smem = cu_seqlens && n_seqs + 1 <= kCuSmemEntries ? 4u * (size_t)(n_seqs + 1) : 0;

  ScalarParams p;
  std::memset(&p, 0, sizeof(p));
  p.br[0].a = a;
  p.br[0].x = x;
  p.br[0].h0 = h0;
  p.br[0].out_h = h;
  p.br[0].dir = reverse ? -1 : 1;
  p.cu = cu_seqlens;
  p.n_seqs = cu_seqlens ? n_seqs : 1;
  p.nbr = 1;
  p.rows = rows;
  p.T = T;
  p.M = (int)M;
  p.G = (int)G;
  p.R = R;
  p.ntiles = tiles;
  p.nseg = 1;
  p.cps = (int)M;
  p.hdr = static_cast<WsHeader*>(scratch);
  p.recs = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(scratch) +
                                                  kWsHeaderBytes);
  p.rec_bytes = need - kWsHeaderBytes;
  p.wait_limit_ns = 1000000000ULL;
  const cudaError_t e = dt == SCAN_F32 ? launch_scalar_fwd_f32(p, pl, stream)
                                       : launch_scalar_fwd_bf16(p, pl, stream);
  return e == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}

extern "C" scan_status scan_noalloc_device_status(cudaStream_t stream) {
  void* scratch = nullptr;
  const scan_status st = scratch_on_current_device(&scratch);
  if (st != SCAN_OK) return st;
  return scan_get_device_status(scratch, stream);
}
