// scan_host.cu -- one forward + backward step of dense rows whose inputs and
// results live in host memory ("Triton scan kernels", the scan and its
// reversed-scan backward; the rows of the dense layout are independent
// recurrences, so any cut between rows is exact).
//
// The rows are cut into pieces. Piece i's inputs are copied to the device on
// one stream, scanned forward and backward on the caller's stream, and its
// results copied back on a third stream; events order each piece's three
// stages, so the copies of neighbouring pieces run under the scans of piece i
// and the two copy directions run at the same time. The scans run one after
// another on the caller's stream, so they share the caller's workspace.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/libscan.h"
#include "scan_internal.h"

namespace scan {
namespace {

constexpr int kMaxPieces = 64;

// Two copy streams and the events of one call, made once per device and
// reused; calls on one device are serialised by the mutex (the events are
// shared).
struct Pipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in_done[kMaxPieces] = {}, scanned[kMaxPieces] = {};
  bool ready = false;
};

std::mutex g_mu;
std::vector<Pipe> g_pipes;

cudaError_t make_pipe(Pipe& p) {
  cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.end, cudaEventDisableTiming);
  for (int i = 0; i < kMaxPieces && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&p.in_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.scanned[i], cudaEventDisableTiming);
  }
  p.ready = e == cudaSuccess;
  return e;
}

const char* cbyte(const void* p, int64_t off) { return static_cast<const char*>(p) + off; }
char* byte(void* p, int64_t off) { return static_cast<char*>(p) + off; }

}  // namespace
}  // namespace scan

using namespace scan;

extern "C" scan_status scan_step_host(const scan_host_io* host, const scan_device_io* dev,
                                      int64_t B, int64_t C, int64_t T, scan_dtype dt,
                                      int32_t pieces, const scan_opts* opts, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
  if (!host || !dev || B < 0 || C < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  if (pieces < 0 || pieces > kMaxPieces) return SCAN_ERR_INVALID_ARG;
  const int64_t rows = B * C;
  if (rows * T == 0) return SCAN_OK;
  if (!host->a || !host->x || !host->dh || !host->h || !host->da || !host->dx)
    return SCAN_ERR_INVALID_ARG;
  if (!dev->a || !dev->x || !dev->dh || !dev->h || !dev->da || !dev->dx) return SCAN_ERR_INVALID_ARG;
  // h0 and dh0 are optional, but on both sides or on neither
  if ((host->h0 == nullptr) != (dev->h0 == nullptr)) return SCAN_ERR_INVALID_ARG;
  if ((host->dh0 == nullptr) != (dev->dh0 == nullptr)) return SCAN_ERR_INVALID_ARG;

  scan_opts o{};
  if (opts) o = *opts;
  // a piece holds fewer rows than the GPU has warp slots; the scans keep the
  // register carry (no per-chunk summaries) unless the caller says otherwise
  if (o.variant == SCAN_VARIANT_AUTO) o.variant = SCAN_VARIANT_STATIONARY;
  const int np = (int)(pieces == 0 ? (rows < 8 ? rows : 8) : (pieces < rows ? pieces : rows));
  const int64_t esz = dt == SCAN_F32 ? 4 : 2;
  // The plans of the largest piece are checked before anything is queued, so
  // a call rejected for its options or its workspace leaves nothing in flight
  // (a smaller piece needs no more workspace than the largest).
  const int64_t big = (rows + np - 1) / np;
  const scan_status ps = scalar_plan_status(big, T, 1, &o);
  if (ps != SCAN_OK) return ps;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SCAN_ERR_WORKSPACE;
  for (scan_op op : {SCAN_OP_FWD, SCAN_OP_BWD})
    if (workspace_bytes < scan_workspace_bytes(op, 1, big, T, 0, 0, &o)) return SCAN_ERR_WORKSPACE;

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SCAN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if ((int)g_pipes.size() <= device) g_pipes.resize(device + 1);
  Pipe& pp = g_pipes[device];
  if (!pp.ready && make_pipe(pp) != cudaSuccess) return SCAN_ERR_CUDA;

  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // on a failure after the first copy was queued, the caller's stream still
  // waits for the copies in flight (best effort) before the status returns
  auto fail = [&](scan_status st) {
    if (ok(cudaEventRecord(pp.end, pp.in))) cudaStreamWaitEvent(stream, pp.end, 0);
    if (ok(cudaEventRecord(pp.end, pp.out))) cudaStreamWaitEvent(stream, pp.end, 0);
    return st;
  };
  // the copies start after the work already queued on the caller's stream
  if (!ok(cudaEventRecord(pp.start, stream)) || !ok(cudaStreamWaitEvent(pp.in, pp.start, 0)) ||
      !ok(cudaStreamWaitEvent(pp.out, pp.start, 0)))
    return SCAN_ERR_CUDA;

  for (int i = 0; i < np; ++i) {
    const int64_t r0 = rows * i / np, r1 = rows * (i + 1) / np, n = r1 - r0;
    const int64_t lo = r0 * T * esz, nb = n * T * esz;    // a, x, da, dx
    const int64_t lo4 = r0 * T * 4, nb4 = n * T * 4;      // dh, h (fp32)
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    // ---- in ----
    if (!ok(cudaMemcpyAsync(byte(dev->a, lo), cbyte(host->a, lo), nb, h2d, pp.in)) ||
        !ok(cudaMemcpyAsync(byte(dev->x, lo), cbyte(host->x, lo), nb, h2d, pp.in)) ||
        !ok(cudaMemcpyAsync(byte(dev->dh, lo4), cbyte(host->dh, lo4), nb4, h2d, pp.in)))
      return fail(SCAN_ERR_CUDA);
    if (host->h0 && !ok(cudaMemcpyAsync(dev->h0 + r0, host->h0 + r0, n * 4, h2d, pp.in)))
      return fail(SCAN_ERR_CUDA);
    if (!ok(cudaEventRecord(pp.in_done[i], pp.in))) return fail(SCAN_ERR_CUDA);
    // ---- scans (the caller's stream) ----
    if (!ok(cudaStreamWaitEvent(stream, pp.in_done[i], 0))) return fail(SCAN_ERR_CUDA);
    scan_status st = scan_fwd(cbyte(dev->a, lo), cbyte(dev->x, lo), dev->h0 ? dev->h0 + r0 : nullptr,
                              nullptr, 0, reinterpret_cast<float*>(byte(dev->h, lo4)), 1, n, T, dt,
                              0, &o, workspace, workspace_bytes, stream);
    if (st != SCAN_OK) return fail(st);
    st = scan_bwd(cbyte(dev->a, lo), reinterpret_cast<const float*>(cbyte(dev->h, lo4)),
                  reinterpret_cast<const float*>(cbyte(dev->dh, lo4)),
                  dev->h0 ? dev->h0 + r0 : nullptr, nullptr, 0, byte(dev->da, lo),
                  byte(dev->dx, lo), dev->dh0 ? dev->dh0 + r0 : nullptr, 1, n, T, dt, 0, &o,
                  workspace, workspace_bytes, stream);
    if (st != SCAN_OK) return fail(st);
    if (!ok(cudaEventRecord(pp.scanned[i], stream))) return fail(SCAN_ERR_CUDA);
    // ---- out ----
    if (!ok(cudaStreamWaitEvent(pp.out, pp.scanned[i], 0))) return fail(SCAN_ERR_CUDA);
    if (!ok(cudaMemcpyAsync(byte(host->h, lo4), cbyte(dev->h, lo4), nb4, d2h, pp.out)) ||
        !ok(cudaMemcpyAsync(byte(host->da, lo), cbyte(dev->da, lo), nb, d2h, pp.out)) ||
        !ok(cudaMemcpyAsync(byte(host->dx, lo), cbyte(dev->dx, lo), nb, d2h, pp.out)))
      return fail(SCAN_ERR_CUDA);
    if (host->dh0 && !ok(cudaMemcpyAsync(host->dh0 + r0, dev->dh0 + r0, n * 4, d2h, pp.out)))
      return fail(SCAN_ERR_CUDA);
  }
  // the caller's stream continues after the last copy out
  if (!ok(cudaEventRecord(pp.end, pp.out)) || !ok(cudaStreamWaitEvent(stream, pp.end, 0)))
    return SCAN_ERR_CUDA;
  return SCAN_OK;
}
