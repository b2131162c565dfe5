// scan_api.cu -- the C ABI of libscan: argument checks, the per-shape planner,
// workspace sizing and kernel launches. See include/libscan.h for the contract.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/libscan.h"
#include "scan_internal.h"

using namespace scan;

namespace {

constexpr int64_t kMaxGrid = 0x7fffffffLL;
constexpr int64_t kStationaryMinRows = 152 * 16;
constexpr bool kStreamOutTiles = true;  // stream: interior outputs leave by tensor stores

__global__ void fill_zero_kernel(float* p, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0.f;
}

bool aligned(const void* p, size_t a) { return p == nullptr || ((uintptr_t)p % a) == 0; }

scan_opts defaults(const scan_opts* o) {
  scan_opts d;
  std::memset(&d, 0, sizeof(d));
  if (o) d = *o;
  return d;
}

unsigned long long wait_ns(const scan_opts& o) {
  const double s = o.wait_limit_s > 0 ? o.wait_limit_s : 1.0;
  const double ns = s * 1e9;
  return ns > 1.8e19 ? 18000000000000000000ULL : (unsigned long long)ns;
}

int chunk_to_j(int chunk) {
  switch (chunk) {
    case 128: return 1;
    case 256: return 2;
    case 512: return 4;
    default: return 0;
  }
}

// Per-shape plan for the scalar and log forms. rows = B*C (dense) or C (packed);
// nbr = number of branches launched together.
// wide: rows that prefer chunks of 512 steps on the register-carry kernels:
// dense rows of the linear form's forward (fp32: the interleaved, fully
// coalesced layout; bf16: lane runs of 16 steps), dense fp32 backward rows and
// dense rows of the log form.
// short_runs: stationary rows that prefer chunks of 256 steps even when wide:
// dense fp32 rows of the linear form, whose kernels at that length are held
// to 72 registers (28 row-warps per SM). On 8 x 1536 rows the backward ran
// 0.1651 ms at T = 4096 and 2.516 ms at T = 65536 (chunks of 512 at the
// default budget: 0.1725 and 2.572), the forward 0.1015 / 1.464 ms (0.1014 /
// 1.480).
// r_default: rows per block when the caller leaves it to the planner (dense
// fp32 rows: 2; forward 0.1012 vs 0.1020 ms and backward 0.1694 vs 0.1711 ms
// at 4 rows, at T = 4096).
scan_status plan_scalar(int64_t rows, int64_t T, int nbr, bool varlen, bool wide,
                        const scan_opts& o, ScalarPlan* pl, bool short_runs = false,
                        int r_default = 4) {
  if (rows < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  int variant = o.variant;
  if (variant < 0 || variant > 3) return SCAN_ERR_INVALID_ARG;
  // Stationary blocks walk T in order with the carry in registers and no
  // inter-block traffic; that needs enough rows to occupy every SM (one warp
  // per row, about 16 resident warps per SM on 152 SMs). Fewer rows split T
  // across blocks and use the look-back.
  if (variant == SCAN_VARIANT_AUTO)
    variant = rows * nbr >= kStationaryMinRows ? VAR_STATIONARY : VAR_LOOKBACK;
  // Lane runs of 8 steps (chunks of 256) keep the register-carry kernels'
  // loads at 8 cache lines per warp instruction; wide calls, the stream
  // variant's tiles and the look-back (fewer published summaries per row)
  // take chunks of 512.
  int J;
  if (o.chunk) {
    J = chunk_to_j(o.chunk);
    if (!J) return SCAN_ERR_INVALID_ARG;
  } else if (T <= 256) {
    J = T <= 128 ? 1 : 2;
  } else {
    J = (wide || variant == VAR_LOOKBACK || variant == VAR_STREAM) ? 4 : 2;
    if (short_runs && variant == VAR_STATIONARY) J = 2;
  }
  int R = o.rows_per_cta;
  if (R < 0 || R > 8) return SCAN_ERR_INVALID_ARG;
  if (R == 0) R = rows < r_default ? (int)(rows > 0 ? rows : 1) : r_default;
  const int64_t L = 128LL * J;
  // the vectorised paths shift each row by up to 3 elements (7 for staged
  // bf16 rows)
  const int64_t span = T + ((T % 8) ? 7 : 0);
  const int64_t M = T > 0 ? (span + L - 1) / L : 0;
  const int64_t G = (rows + R - 1) / R;
  const int64_t tiles = M * G * nbr;
  if (M > kMaxGrid || G > kMaxGrid || tiles > kMaxGrid || rows * M * nbr > (1LL << 40))
    return SCAN_ERR_UNSUPPORTED;
  // Stationary rows are cut into segments only on request: a segment cannot
  // start before the end state of the one before it is known, so segments
  // add resident warps that mostly wait (measured slower on every shape the
  // planner sends to STATIONARY).
  int64_t nseg = 1, cps = M;
  if (variant == VAR_STATIONARY && M > 0) {
    if (o.segments < 0) return SCAN_ERR_INVALID_ARG;
    nseg = o.segments ? o.segments : 1;
    if (nseg > M) nseg = M;
    cps = (M + nseg - 1) / nseg;
    nseg = (M + cps - 1) / cps;
    if (nseg * G * nbr > kMaxGrid) return SCAN_ERR_UNSUPPORTED;
  }
  pl->variant = variant;
  pl->J = J;
  pl->R = R;
  pl->M = (int)M;
  pl->G = (int)G;
  pl->nseg = (int)nseg;
  pl->cps = (int)cps;
  pl->vec = true;
  size_t recs = 0;
  if (variant == VAR_LOOKBACK) recs = (size_t)(nbr * rows * M);
  if (variant == VAR_STATIONARY && nseg > 1) recs = (size_t)(nbr * rows * nseg);
  if (o.stages < 0 || o.stages == 1 || o.stages > kMaxStages) return SCAN_ERR_INVALID_ARG;
  pl->ns = o.stages;
  pl->ws_bytes = kWsHeaderBytes + recs * 16u;
  (void)varlen;
  pl->smem = 0;
  return SCAN_OK;
}

// Lane groups of 8 (one warp each) from which the 4 x 4 ring kernel is the
// default: below about one warp per SM the look-back kernels, which split T
// into chunks, keep more of the GPU busy.
constexpr int64_t kAffineRingMinWarps = 152;

// Per-shape plan for the block-matrix form: a block covers 32 / v lanes (one
// thread per column) and one chunk of Lc steps (4 sub-chunks of Lc / 4).
scan_status plan_affine(int64_t B, int64_t T, int64_t N, int k, int v, const scan_opts& o,
                        AffinePlan* pl) {
  if (B < 0 || T < 0 || N < 0) return SCAN_ERR_INVALID_ARG;
  const int rec = affine_record_floats(k, v);
  if (rec == 0) return SCAN_ERR_UNSUPPORTED;
  int Lc = o.chunk ? o.chunk : 64;
  if (Lc != 64 && Lc != 128 && Lc != 256) return SCAN_ERR_INVALID_ARG;
  const int64_t lanes = affine_lanes_per_block(k, v);
  const int64_t M = T > 0 ? (T + Lc - 1) / Lc : 0;
  const int64_t G = B * ((N + lanes - 1) / lanes);
  if (M * G > kMaxGrid) return SCAN_ERR_UNSUPPORTED;
  pl->Lc = Lc;
  pl->M = (int)M;
  pl->G = (int)G;
  // 4 x 4 blocks of lane-rich shapes walk T with the state in registers,
  // fed by a ring of tensor copies (no records, no replay); the rest run the
  // look-back kernels. The workspace is sized for the look-back whatever the
  // variant, so one size serves the coefficient prefix (look-back only) and
  // every option of a shape.
  const bool ring = affine_ring_fits(B, T, N, k, v);
  if (o.variant == SCAN_VARIANT_STATIONARY && ring) pl->variant = VAR_STATIONARY;
  else if (o.variant == SCAN_VARIANT_AUTO && ring && affine_ring_warps(B, N) >= kAffineRingMinWarps)
    pl->variant = VAR_STATIONARY;
  else pl->variant = VAR_LOOKBACK;
  pl->ws_bytes = kWsHeaderBytes + (size_t)(B * N * M) * (size_t)rec * sizeof(float);
  return SCAN_OK;
}

scan_status check_host_cu(const int32_t* cu, int32_t n, int64_t T) {
  if (!cu) return SCAN_OK;
  if (cu[0] != 0 || (int64_t)cu[n] != T) return SCAN_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (cu[i + 1] < cu[i]) return SCAN_ERR_INVALID_ARG;
  return SCAN_OK;
}

// Shared front end of the scalar/log entry points: shape checks, plan,
// workspace check, base parameters.
scan_status prepare(int64_t B, int64_t C, int64_t T, const int32_t* cu, int32_t n_seqs, int nbr,
                    bool wide, const scan_opts& o, void* ws, size_t ws_bytes,
                    ScalarParams* p, ScalarPlan* pl, bool short_runs = false,
                    int r_default = 4) {
  if (B < 0 || C < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (cu) {
    if (B != 1 || n_seqs < 1 || T > 0x7fffffffLL) return SCAN_ERR_INVALID_ARG;
    if (o.cu_seqlens_host) {
      const scan_status st = check_host_cu(o.cu_seqlens_host, n_seqs, T);
      if (st != SCAN_OK) return st;
    }
  }
  const int64_t rows = B * C;
  scan_status st = plan_scalar(rows, T, nbr, cu != nullptr, wide, o, pl, short_runs, r_default);
  if (st != SCAN_OK) return st;
  if (!ws) return SCAN_ERR_WORKSPACE;
  if (ws_bytes < pl->ws_bytes || !aligned(ws, 16)) return SCAN_ERR_WORKSPACE;
  // packed offsets are staged in shared memory when they fit
  if (cu) pl->smem = n_seqs + 1 <= kCuSmemEntries ? 4u * (size_t)(n_seqs + 1) : 0u;
  std::memset(p, 0, sizeof(*p));
  p->cu = cu;
  p->n_seqs = cu ? n_seqs : 1;
  p->nbr = nbr;
  p->rows = rows;
  p->T = T;
  p->M = pl->M;
  p->G = pl->G;
  p->R = pl->R;
  p->nseg = pl->nseg;
  p->cps = pl->cps;
  p->ntiles = (pl->variant == VAR_LOOKBACK ? (int64_t)pl->M : (int64_t)pl->nseg) * pl->G * nbr;
  p->hdr = static_cast<WsHeader*>(ws);
  p->recs = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(ws) +
                                                  kWsHeaderBytes);
  p->rec_bytes = pl->ws_bytes - kWsHeaderBytes;
  p->wait_limit_ns = wait_ns(o);
  p->test_stall = o.test_stall;
  return SCAN_OK;
}

// Workspace of a scalar/log call: the larger of the two layouts' plans, so
// one size serves every dtype and form of the call.
size_t ws_scalar(int64_t rows, int64_t T, int nbr, const scan_opts& o) {
  ScalarPlan a, b;
  if (plan_scalar(rows, T, nbr, false, false, o, &a) != SCAN_OK) return 0;
  if (plan_scalar(rows, T, nbr, false, true, o, &b) != SCAN_OK) return 0;
  return a.ws_bytes > b.ws_bytes ? a.ws_bytes : b.ws_bytes;
}

// The stream variant reads and writes every tensor through tensor maps: all
// of them 16-byte aligned, at least one 128-byte row (64 elements) long, and
// a ring that fits in shared memory; otherwise the same rows run STATIONARY.
// Its chunks start on a 128-byte row of the flat tensor, so a row is shifted
// by up to E - 1 elements (E = 128 / element size of a) and M is recounted;
// without segments it needs only the workspace header.
void finish_plan(ScalarPlan* pl, ScalarParams* p, int mode, int elt_a, bool all16,
                 int rows_per_cta) {
  if (pl->variant != VAR_STREAM) return;
  const int E = tma_row_elems(elt_a);
  const int64_t n = p->rows * p->T;
  auto fallback = [&] {
    pl->variant = VAR_STATIONARY;
    pl->nseg = p->nseg = 1;
    pl->cps = p->cps = pl->M;
  };
  if (!pl->vec || !all16 || n < E) return fallback();
  if (rows_per_cta == 0) {
    pl->R = p->R = 1;
    pl->G = p->G = (int)((p->rows + pl->R - 1) / pl->R);
  }
  const int64_t L = 128LL * pl->J;
  const int64_t span = p->T + ((p->T % E) ? E - 1 : 0);
  pl->M = p->M = (int)((span + L - 1) / L);
  // the stage is refilled as soon as it is in registers, so a few stages
  // cover the copies' latency
  const int ns = pl->ns ? pl->ns : 3;
  pl->tma_out = kStreamOutTiles;
  const size_t cu = round_up(pl->smem, 128);
  auto total = [&](int k) {
    return cu + tma_bar_bytes(pl->R) + 1024 +
           (size_t)pl->R * tma_warp_bytes(mode, pl->J, elt_a, k, pl->tma_out);
  };
  if (total(ns) > 227 * 1024) return fallback();
  pl->ns = p->ns = ns;
  p->tma_out = pl->tma_out ? 1 : 0;
  pl->nseg = p->nseg = 1;
  pl->cps = p->cps = pl->M;
  pl->smem = total(ns);
}

scan_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA; }

// dh0 when there is nothing to scan: every initial-state gradient is 0.
scan_status zero_dh0(float* dh0, int64_t n, cudaStream_t s) {
  if (!dh0 || n <= 0) return SCAN_OK;
  return from_cuda(launch_fill_zero(dh0, n, s));
}

size_t elt(scan_dtype dt) { return dt == SCAN_BF16 ? 2 : 4; }

}  // namespace

namespace scan {
scan_status scalar_plan_status(int64_t rows, int64_t T, int nbr, const scan_opts* opts) {
  const scan_opts o = defaults(opts);
  for (int w = 0; w < 2; ++w)
    for (int sr = 0; sr < 2; ++sr) {
      ScalarPlan pl;
      const scan_status st = plan_scalar(rows, T, nbr, false, w != 0, o, &pl, sr != 0);
      if (st != SCAN_OK) return st;
    }
  return SCAN_OK;
}

cudaError_t launch_fill_zero(float* p, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
  fill_zero_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, n);
  return cudaGetLastError();
}
}  // namespace scan

extern "C" {

const char* scan_status_string(scan_status s) {
  switch (s) {
    case SCAN_OK: return "SCAN_OK";
    case SCAN_ERR_INVALID_ARG: return "SCAN_ERR_INVALID_ARG: malformed argument";
    case SCAN_ERR_UNSUPPORTED: return "SCAN_ERR_UNSUPPORTED: outside the supported envelope";
    case SCAN_ERR_ALIGNMENT: return "SCAN_ERR_ALIGNMENT: misaligned pointer";
    case SCAN_ERR_WORKSPACE: return "SCAN_ERR_WORKSPACE: workspace missing or too small";
    case SCAN_ERR_CUDA: return "SCAN_ERR_CUDA: CUDA runtime error";
    case SCAN_ERR_TIMEOUT: return "SCAN_ERR_TIMEOUT: a look-back wait expired on the device";
    case SCAN_ERR_SEQLENS: return "SCAN_ERR_SEQLENS: cu_seqlens is not 0 <= ... <= T";
    default: return "unknown scan_status";
  }
}

int32_t scan_version(void) { return LIBSCAN_VERSION; }

size_t scan_workspace_bytes(scan_op op, int64_t B, int64_t C, int64_t T, int32_t k, int32_t v,
                            const scan_opts* opts) {
  const scan_opts o = defaults(opts);
  if (B < 0 || C < 0 || T < 0) return 0;
  switch (op) {
    case SCAN_OP_FWD:
    case SCAN_OP_BWD:
    case SCAN_OP_LOG_FWD:
    case SCAN_OP_LOG_BWD:
      return ws_scalar(B * C, T, 1, o);
    case SCAN_OP_BIDIR_FWD:
    case SCAN_OP_BIDIR_BWD:
      return ws_scalar(B * C, T, 2, o);
    case SCAN_OP_AFFINE_FWD:
    case SCAN_OP_AFFINE_BWD: {
      AffinePlan ap;
      return plan_affine(B, T, C, k, v, o, &ap) == SCAN_OK ? ap.ws_bytes : 0;
    }
    default:
      return 0;
  }
}

scan_status scan_workspace_init(void* ws, size_t bytes, cudaStream_t stream) {
  if (!ws || bytes < kWsHeaderBytes) return SCAN_ERR_WORKSPACE;
  return from_cuda(cudaMemsetAsync(ws, 0, bytes, stream));
}

scan_status scan_get_device_status(void* ws, cudaStream_t stream) {
  if (!ws) return SCAN_ERR_WORKSPACE;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SCAN_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return SCAN_ERR_CUDA;
  if (h.status != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(static_cast<unsigned char*>(ws) + offsetof(WsHeader, status), &zero,
                   sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return SCAN_ERR_CUDA;
  }
  return (scan_status)h.status;
}

scan_status scan_fwd(const void* a, const void* x, const float* h0, const int32_t* cu,
                     int32_t n_seqs, float* h, int64_t B, int64_t C, int64_t T, scan_dtype dt,
                     int32_t reverse, const scan_opts* opts, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  const scan_opts o = defaults(opts);
  ScalarParams p;
  ScalarPlan pl;
  // dense bf16 rows: lane runs of 16 steps, one row per block (8 x 1536 x
  // 4096: 0.0900 vs 0.0996 ms at runs of 8 and 4 rows per block)
  const bool dense32 = !cu && dt == SCAN_F32;
  scan_status st = prepare(B, C, T, cu, n_seqs, 1, !cu, o, ws, ws_bytes, &p, &pl, dense32,
                           dense32 ? 2 : (cu ? 4 : 1));
  if (st != SCAN_OK) return st;
  if (p.rows * T == 0) return SCAN_OK;
  if (!a || !x || !h) return SCAN_ERR_INVALID_ARG;
  pl.vec = aligned(a, 4 * elt(dt)) && aligned(x, 4 * elt(dt)) && aligned(h, 16);
  finish_plan(&pl, &p, MODE_FWD, (int)elt(dt), aligned(a, 16) && aligned(x, 16) && aligned(h, 16),
              o.rows_per_cta);
  p.br[0].a = a;
  p.br[0].x = x;
  p.br[0].h0 = h0;
  p.br[0].out_h = h;
  p.br[0].dir = reverse ? -1 : 1;
  return from_cuda(dt == SCAN_F32 ? launch_scalar_fwd_f32(p, pl, stream)
                                  : launch_scalar_fwd_bf16(p, pl, stream));
}

scan_status scan_bwd(const void* a, const float* h, const float* dh, const float* h0,
                     const int32_t* cu, int32_t n_seqs, void* da, void* dx, float* dh0,
                     int64_t B, int64_t C, int64_t T, scan_dtype dt, int32_t reverse,
                     const scan_opts* opts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  const scan_opts o = defaults(opts);
  ScalarParams p;
  ScalarPlan pl;
  // dense bf16 rows keep runs of 8 (16: 0.163 vs 0.137 ms on 8 x 1536 x
  // 4096), two rows per block (4: 0.1382 ms)
  const bool dense32 = !cu && dt == SCAN_F32;
  scan_status st = prepare(B, C, T, cu, n_seqs, 1, dense32, o, ws, ws_bytes, &p, &pl, dense32,
                           cu ? 4 : 2);
  if (st != SCAN_OK) return st;
  const int64_t n_h0 = cu ? (int64_t)n_seqs * C : B * C;
  if (p.rows * T == 0) return zero_dh0(dh0, n_h0, stream);
  if (!a || !h || !dh || !da || !dx) return SCAN_ERR_INVALID_ARG;
  pl.vec = aligned(a, 4 * elt(dt)) && aligned(da, 4 * elt(dt)) && aligned(dx, 4 * elt(dt)) &&
           aligned(h, 16) && aligned(dh, 16);
  finish_plan(&pl, &p, MODE_BWD, (int)elt(dt),
              aligned(a, 16) && aligned(h, 16) && aligned(dh, 16) && aligned(da, 16) &&
                  aligned(dx, 16),
              o.rows_per_cta);
  p.br[0].a = a;
  p.br[0].h = h;
  p.br[0].dh = dh;
  p.br[0].h0 = h0;
  p.br[0].da = da;
  p.br[0].dx = dx;
  p.br[0].dh0 = dh0;
  p.br[0].dir = reverse ? -1 : 1;
  return from_cuda(dt == SCAN_F32 ? launch_scalar_bwd_f32(p, pl, stream)
                                  : launch_scalar_bwd_bf16(p, pl, stream));
}

scan_status scan_bidir_fwd(const void* af, const void* xf, const void* ar, const void* xr,
                           const float* h0f, const float* h0r, const int32_t* cu, int32_t n_seqs,
                           float* hf, float* hr, int64_t B, int64_t C, int64_t T, scan_dtype dt,
                           const scan_opts* opts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  const scan_opts o = defaults(opts);
  ScalarParams p;
  ScalarPlan pl;
  scan_status st =
      prepare(B, C, T, cu, n_seqs, 2, !cu && dt == SCAN_F32, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  if (p.rows * T == 0) return SCAN_OK;
  if (!af || !xf || !ar || !xr || !hf || !hr) return SCAN_ERR_INVALID_ARG;
  const size_t va = 4 * elt(dt);
  pl.vec = aligned(af, va) && aligned(xf, va) && aligned(ar, va) && aligned(xr, va) &&
           aligned(hf, 16) && aligned(hr, 16);
  finish_plan(&pl, &p, MODE_FWD, (int)elt(dt),
              aligned(af, 16) && aligned(xf, 16) && aligned(ar, 16) && aligned(xr, 16) &&
                  aligned(hf, 16) && aligned(hr, 16),
              o.rows_per_cta);
  p.br[0].a = af;
  p.br[0].x = xf;
  p.br[0].h0 = h0f;
  p.br[0].out_h = hf;
  p.br[0].dir = 1;
  p.br[1].a = ar;
  p.br[1].x = xr;
  p.br[1].h0 = h0r;
  p.br[1].out_h = hr;
  p.br[1].dir = -1;
  return from_cuda(dt == SCAN_F32 ? launch_scalar_fwd_f32(p, pl, stream)
                                  : launch_scalar_fwd_bf16(p, pl, stream));
}

scan_status scan_bidir_bwd(const void* af, const float* hf, const float* dhf, const float* h0f,
                           const void* ar, const float* hr, const float* dhr, const float* h0r,
                           const int32_t* cu, int32_t n_seqs, void* daf, void* dxf, float* dh0f,
                           void* dar, void* dxr, float* dh0r, int64_t B, int64_t C, int64_t T,
                           scan_dtype dt, const scan_opts* opts, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  const scan_opts o = defaults(opts);
  ScalarParams p;
  ScalarPlan pl;
  scan_status st =
      prepare(B, C, T, cu, n_seqs, 2, !cu && dt == SCAN_F32, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  const int64_t n_h0 = cu ? (int64_t)n_seqs * C : B * C;
  if (p.rows * T == 0) {
    st = zero_dh0(dh0f, n_h0, stream);
    return st != SCAN_OK ? st : zero_dh0(dh0r, n_h0, stream);
  }
  if (!af || !hf || !dhf || !ar || !hr || !dhr || !daf || !dxf || !dar || !dxr)
    return SCAN_ERR_INVALID_ARG;
  const size_t va = 4 * elt(dt);
  pl.vec = aligned(af, va) && aligned(ar, va) && aligned(daf, va) && aligned(dxf, va) &&
           aligned(dar, va) && aligned(dxr, va) && aligned(hf, 16) && aligned(dhf, 16) &&
           aligned(hr, 16) && aligned(dhr, 16);
  finish_plan(&pl, &p, MODE_BWD, (int)elt(dt),
              aligned(af, 16) && aligned(ar, 16) && aligned(hf, 16) && aligned(dhf, 16) &&
                  aligned(hr, 16) && aligned(dhr, 16) && aligned(daf, 16) && aligned(dxf, 16) &&
                  aligned(dar, 16) && aligned(dxr, 16),
              o.rows_per_cta);
  p.br[0].a = af;
  p.br[0].h = hf;
  p.br[0].dh = dhf;
  p.br[0].h0 = h0f;
  p.br[0].da = daf;
  p.br[0].dx = dxf;
  p.br[0].dh0 = dh0f;
  p.br[0].dir = 1;
  p.br[1].a = ar;
  p.br[1].h = hr;
  p.br[1].dh = dhr;
  p.br[1].h0 = h0r;
  p.br[1].da = dar;
  p.br[1].dx = dxr;
  p.br[1].dh0 = dh0r;
  p.br[1].dir = -1;
  return from_cuda(dt == SCAN_F32 ? launch_scalar_bwd_f32(p, pl, stream)
                                  : launch_scalar_bwd_bf16(p, pl, stream));
}

scan_status scan_log_fwd(const float* log_a, const float* log_x, const float* log_h0,
                         const int32_t* cu, int32_t n_seqs, float* h, int64_t B, int64_t C,
                         int64_t T, int32_t reverse, const scan_opts* opts, void* ws,
                         size_t ws_bytes, cudaStream_t stream) {
  const scan_opts o = defaults(opts);
  ScalarParams p;
  ScalarPlan pl;
  // dense rows: 16-step lane runs halve the per-run share of the warp scan,
  // which is costly in log space (measured 7 % faster than 8-step runs)
  scan_status st = prepare(B, C, T, cu, n_seqs, 1, !cu, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  if (p.rows * T == 0) return SCAN_OK;
  if (!log_a || !log_x || !h) return SCAN_ERR_INVALID_ARG;
  pl.vec = aligned(log_a, 16) && aligned(log_x, 16) && aligned(h, 16);
  finish_plan(&pl, &p, MODE_FWD, 4, aligned(log_a, 16) && aligned(log_x, 16) && aligned(h, 16),
              o.rows_per_cta);
  p.br[0].a = log_a;
  p.br[0].x = log_x;
  p.br[0].h0 = log_h0;
  p.br[0].out_h = h;
  p.br[0].dir = reverse ? -1 : 1;
  return from_cuda(launch_log_fwd(p, pl, stream));
}

scan_status scan_log_bwd(const float* log_a, const float* log_x, const float* h, const float* dh,
                         const float* log_h0, const int32_t* cu, int32_t n_seqs, float* dlog_a,
                         float* dlog_x, float* dlog_h0, int64_t B, int64_t C, int64_t T,
                         int32_t reverse, const scan_opts* opts, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  scan_opts o = defaults(opts);
  if (o.variant == SCAN_VARIANT_STREAM) o.variant = SCAN_VARIANT_STATIONARY;
  ScalarParams p;
  ScalarPlan pl;
  scan_status st = prepare(B, C, T, cu, n_seqs, 1, false, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  const int64_t n_h0 = cu ? (int64_t)n_seqs * C : B * C;
  if (p.rows * T == 0) return zero_dh0(dlog_h0, n_h0, stream);
  if (!log_a || !log_x || !h || !dh || !dlog_a || !dlog_x) return SCAN_ERR_INVALID_ARG;
  pl.vec = aligned(log_a, 16) && aligned(log_x, 16) && aligned(h, 16) && aligned(dh, 16) &&
           aligned(dlog_a, 16) && aligned(dlog_x, 16);
  p.br[0].a = log_a;
  p.br[0].x = log_x;
  p.br[0].h = h;
  p.br[0].dh = dh;
  p.br[0].h0 = log_h0;
  p.br[0].da = dlog_a;
  p.br[0].dx = dlog_x;
  p.br[0].dh0 = dlog_h0;
  p.br[0].dir = reverse ? -1 : 1;
  return from_cuda(launch_log_bwd(p, pl, stream));
}

}  // extern "C"

namespace {

scan_status prepare_affine(int64_t B, int64_t T, int64_t N, int32_t k, int32_t v,
                           const scan_opts& o, void* ws, size_t ws_bytes, AffineParams* p,
                           AffinePlan* pl) {
  scan_status st = plan_affine(B, T, N, k, v, o, pl);
  if (st != SCAN_OK) return st;
  if (!ws || ws_bytes < pl->ws_bytes || !aligned(ws, 16)) return SCAN_ERR_WORKSPACE;
  std::memset(p, 0, sizeof(*p));
  p->B = B;
  p->T = T;
  p->N = N;
  p->k = k;
  p->v = v;
  p->Lc = pl->Lc;
  p->M = pl->M;
  p->G = pl->G;
  p->ntiles = (int64_t)pl->M * pl->G;
  p->hdr = static_cast<WsHeader*>(ws);
  p->recs = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kWsHeaderBytes);
  p->rec_bytes = pl->ws_bytes - kWsHeaderBytes;
  p->wait_limit_ns = wait_ns(o);
  p->test_stall = o.test_stall;
  return SCAN_OK;
}

}  // namespace

extern "C" {

scan_status affine_scan_fwd(const float* A, const float* Bm, const float* h0, float* H, int64_t B,
                            int64_t T, int64_t N, int32_t k, int32_t v, const scan_opts* opts,
                            void* ws, size_t ws_bytes, cudaStream_t stream) {
  const scan_opts o = defaults(opts);
  AffineParams p;
  AffinePlan pl;
  scan_status st = prepare_affine(B, T, N, k, v, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  if (B * T * N == 0) return SCAN_OK;
  if (!A || !Bm || !H) return SCAN_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(Bm, 16) || !aligned(H, 16) || !aligned(h0, 16))
    return SCAN_ERR_ALIGNMENT;
  p.A = A;
  p.Bm = Bm;
  p.h0 = h0;
  p.out_H = H;
  return from_cuda(launch_affine_fwd(p, pl, stream));
}

scan_status affine_scan_bwd(const float* A, const float* H, const float* dH, const float* h0,
                            float* dA, float* dB, float* dh0, int64_t B, int64_t T, int64_t N,
                            int32_t k, int32_t v, const scan_opts* opts, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  const scan_opts o = defaults(opts);
  AffineParams p;
  AffinePlan pl;
  scan_status st = prepare_affine(B, T, N, k, v, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  if (B * N == 0) return SCAN_OK;
  if (T == 0) return zero_dh0(dh0, B * N * (int64_t)k * v, stream);
  if (!A || !H || !dH || !dA || !dB) return SCAN_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(H, 16) || !aligned(dH, 16) || !aligned(dA, 16) ||
      !aligned(dB, 16) || !aligned(h0, 16) || !aligned(dh0, 16))
    return SCAN_ERR_ALIGNMENT;
  p.A = A;
  p.H = H;
  p.dH = dH;
  p.h0 = h0;
  p.dA = dA;
  p.dB = dB;
  p.dh0 = dh0;
  return from_cuda(launch_affine_bwd(p, pl, stream));
}

scan_status affine_prefix_fwd(const float* A, float* Abar, int64_t B, int64_t T, int64_t N,
                              int32_t k, const scan_opts* opts, void* ws, size_t ws_bytes,
                              cudaStream_t stream) {
  const scan_opts o = defaults(opts);
  AffineParams p;
  AffinePlan pl;
  scan_status st = prepare_affine(B, T, N, k, k, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  if (B * T * N == 0) return SCAN_OK;
  if (!A || !Abar) return SCAN_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(Abar, 16)) return SCAN_ERR_ALIGNMENT;
  p.A = A;
  p.out_H = Abar;
  p.flags = AFF_ZERO_B | AFF_EYE_H0;
  return from_cuda(launch_affine_fwd(p, pl, stream));
}

scan_status affine_prefix_bwd(const float* A, const float* Abar, const float* dAbar, float* dA,
                              int32_t accumulate, int64_t B, int64_t T, int64_t N, int32_t k,
                              const scan_opts* opts, void* ws, size_t ws_bytes,
                              cudaStream_t stream) {
  const scan_opts o = defaults(opts);
  AffineParams p;
  AffinePlan pl;
  scan_status st = prepare_affine(B, T, N, k, k, o, ws, ws_bytes, &p, &pl);
  if (st != SCAN_OK) return st;
  if (B * T * N == 0) return SCAN_OK;
  if (!A || !Abar || !dAbar || !dA) return SCAN_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(Abar, 16) || !aligned(dAbar, 16) || !aligned(dA, 16))
    return SCAN_ERR_ALIGNMENT;
  p.A = A;
  p.H = Abar;
  p.dH = dAbar;
  p.dA = dA;
  p.flags = AFF_EYE_H0 | (accumulate ? AFF_ACC_DA : 0);
  return from_cuda(launch_affine_bwd(p, pl, stream));
}

}  // extern "C"
