// scan_gdn.cu -- the scalar-gated outer-product state ("Operations & Triton
// Kernels" (HyMo), The chunked GDN algorithm; Mathematical Derivation of the
// Reverse-Time Backward Pass):
//   h_t = alpha_t h_{t-1} + b_t v_t^T      (S x D state per (batch, head))
//   o_t = h_t^T c_t                         (D-vector)
// and its reverse-time backward with the states recomputed from checkpoints.
//
// Work decomposition: one warp per (batch, head) walks T with the state in
// registers, lane d holding column d of h (S values). The per-step inputs
// (b_t, c_t: read by every lane; v_t: one element per lane) are staged in
// shared memory by asynchronous 16-byte copies, 32 steps per stage, two
// stages in flight. The forward stores the state before every 64th step
// (the checkpoints the backward starts from). The backward walks those 64-step
// blocks from the end: it stages the block's inputs, recomputes the block's
// states forward keeping the one before every 16th step, and then, for each
// 16-step piece from the last, recomputes its 16 states into shared memory and
// runs the adjoint over them: dh_t = c_t do_t^T + alpha_{t+1} dh_{t+1},
// dv_t = dh_t^T b_t (per lane), db_t = dh_t v_t and dc_t = h_t do_t (summed
// over the lanes by a reduce-scatter of shuffles), dalpha_t = <dh_t, h_{t-1}>.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/libscan.h"
#include "scan_internal.h"

namespace scan {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kStage = 32;  // forward: steps per staged block
constexpr int kCoarse = 64;  // checkpoint interval
constexpr int kFine = 16;    // backward: states recomputed at a time

struct GdnParams {
  const float* alpha;  // [B,H,T]
  const float* b;      // [B,H,T,S]
  const float* v;      // [B,H,T,D]
  const float* c;      // [B,H,T,S]
  const float* h0;     // [B,H,S,D] nullable
  float* o;            // forward output [B,H,T,D]
  float* ckpt;         // [B,H,NC,S,D], NC = ceil(T / 64): state before step 64 j
  const float* dout;   // backward
  float* dalpha;
  float* db;
  float* dv;
  float* dc;
  float* dh0;          // nullable
  int64_t BH, T;
  int64_t NC;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copies `rows` rows of `width` floats (width % 4 == 0) from src to dst with the
// warp's 32 lanes, 16 bytes per copy.
__device__ __forceinline__ void stage_rows(float* dst, const float* src, int rows, int width,
                                           int lane) {
  const int n = rows * width / 4;
  for (int i = lane; i < n; i += 32) cp_async16(dst + 4 * i, src + 4 * i);
}

// Sum over the 32 lanes of 32 per-lane values x[0..31]: afterwards lane j
// holds the total of x[j]. Recursive halving: at each round a lane keeps the
// half of its values selected by its lane bit and adds the partner's copy.
__device__ __forceinline__ float reduce_scatter32(float (&x)[32], int lane) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      // slots i (low half) and i + m (high half) of the current 2m values
      const float send = hi ? x[i] : x[i + m];
      const float keep = hi ? x[i + m] : x[i];
      x[i] = keep + __shfl_xor_sync(kFullMask, send, m);
    }
  }
  return x[0];
}

template <int S, int D>
__global__ void __launch_bounds__(32) gdn_fwd_kernel(const GdnParams p) {
  __shared__ __align__(16) float s_b[2][kStage * S];
  __shared__ __align__(16) float s_c[2][kStage * S];
  __shared__ __align__(16) float s_v[2][kStage * D];
  const int lane = threadIdx.x;
  const int64_t bh = blockIdx.x;
  if (bh >= p.BH) return;
  const int64_t T = p.T;
  const int d = lane < D ? lane : 0;
  const bool col = lane < D;
  float h[S];
#pragma unroll
  for (int s = 0; s < S; ++s) h[s] = (p.h0 && col) ? p.h0[(bh * S + s) * D + d] : 0.f;

  const float* gb = p.b + bh * T * S;
  const float* gc = p.c + bh * T * S;
  const float* gv = p.v + bh * T * D;
  const int nblk = (int)((T + kStage - 1) / kStage);
  auto issue = [&](int blk) {
    const int64_t t0 = (int64_t)blk * kStage;
    const int rows = (int)(T - t0 < kStage ? T - t0 : kStage);
    const int st = blk & 1;
    stage_rows(s_b[st], gb + t0 * S, rows, S, lane);
    stage_rows(s_c[st], gc + t0 * S, rows, S, lane);
    stage_rows(s_v[st], gv + t0 * D, rows, D, lane);
    cp_async_commit();
  };
  issue(0);
  for (int blk = 0; blk < nblk; ++blk) {
    if (blk + 1 < nblk) {
      issue(blk + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const int st = blk & 1;
    const int64_t t0 = (int64_t)blk * kStage;
    const int rows = (int)(T - t0 < kStage ? T - t0 : kStage);
    const float al_lane = lane < rows ? __ldg(p.alpha + bh * T + t0 + lane) : 0.f;
    for (int r = 0; r < rows; ++r) {
      const int64_t t = t0 + r;
      if (p.ckpt && (t % kCoarse) == 0 && col) {
        float* ck = p.ckpt + (bh * p.NC + t / kCoarse) * S * D;
#pragma unroll
        for (int s = 0; s < S; ++s) ck[s * D + d] = h[s];
      }
      const float al = __shfl_sync(kFullMask, al_lane, r);
      const float vd = s_v[st][r * D + d];
      const float* br = s_b[st] + r * S;
      const float* cr = s_c[st] + r * S;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < S; s += 4) {
        const float4 bq = *reinterpret_cast<const float4*>(br + s);
        const float4 cq = *reinterpret_cast<const float4*>(cr + s);
        h[s] = fmaf(al, h[s], bq.x * vd);
        h[s + 1] = fmaf(al, h[s + 1], bq.y * vd);
        h[s + 2] = fmaf(al, h[s + 2], bq.z * vd);
        h[s + 3] = fmaf(al, h[s + 3], bq.w * vd);
        acc[0] = fmaf(cq.x, h[s], acc[0]);
        acc[1] = fmaf(cq.y, h[s + 1], acc[1]);
        acc[2] = fmaf(cq.z, h[s + 2], acc[2]);
        acc[3] = fmaf(cq.w, h[s + 3], acc[3]);
      }
      if (col) __stcs(p.o + (bh * T + t) * D + d, (acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
    __syncwarp();  // the stage is refilled two blocks later
  }
}

template <int S, int D>
__global__ void __launch_bounds__(32) gdn_bwd_kernel(const GdnParams p) {
  extern __shared__ __align__(16) float sm[];
  // inputs of one 64-step block, the states before each 16-step piece, and
  // the 16 states of the current piece
  float* s_b = sm;                        // [64][S]
  float* s_c = s_b + kCoarse * S;         // [64][S]
  float* s_v = s_c + kCoarse * S;         // [64][D]
  float* s_do = s_v + kCoarse * D;        // [64][D]
  float* s_al = s_do + kCoarse * D;       // [65]: alpha of the block's steps and of the next step
  float* s_fine = s_al + kCoarse + 4;     // [4][S][D]
  float* s_st = s_fine + 4 * S * D;       // [16][S][D]
  const int lane = threadIdx.x;
  const int64_t bh = blockIdx.x;
  if (bh >= p.BH) return;
  const int64_t T = p.T;
  const int d = lane < D ? lane : 0;
  const bool col = lane < D;

  float dh[S];
#pragma unroll
  for (int s = 0; s < S; ++s) dh[s] = 0.f;

  for (int64_t J = p.NC - 1; J >= 0; --J) {
    const int64_t t0 = J * kCoarse;
    const int rows = (int)(T - t0 < kCoarse ? T - t0 : kCoarse);
    // ---- stage the block's inputs ----
    stage_rows(s_b, p.b + (bh * T + t0) * S, rows, S, lane);
    stage_rows(s_c, p.c + (bh * T + t0) * S, rows, S, lane);
    stage_rows(s_v, p.v + (bh * T + t0) * D, rows, D, lane);
    stage_rows(s_do, p.dout + (bh * T + t0) * D, rows, D, lane);
    cp_async_commit();
    for (int i = lane; i <= rows; i += 32) {
      const int64_t t = t0 + i;
      s_al[i] = t < T ? __ldg(p.alpha + bh * T + t) : 0.f;  // alpha_{T} = 0 past the end
    }
    // ---- the states before each 16-step piece, from the checkpoint ----
    float h[S];
#pragma unroll
    for (int s = 0; s < S; ++s) h[s] = col ? p.ckpt[(bh * p.NC + J) * S * D + s * D + d] : 0.f;
    cp_async_wait<0>();
    __syncwarp();
    const int npiece = (rows + kFine - 1) / kFine;
    const int last_start = (npiece - 1) * kFine;  // no step after it is needed here
    for (int r = 0;; ++r) {
      if (r % kFine == 0 && col) {
#pragma unroll
        for (int s = 0; s < S; ++s) s_fine[((r / kFine) * S + s) * D + d] = h[s];
      }
      if (r == last_start) break;
      const float al = s_al[r];
      const float vd = s_v[r * D + d];
#pragma unroll
      for (int s = 0; s < S; ++s) h[s] = fmaf(al, h[s], s_b[r * S + s] * vd);
    }
    __syncwarp();
    // ---- pieces from the last: recompute 16 states, then the adjoint ----
    for (int f = npiece - 1; f >= 0; --f) {
      const int r0 = f * kFine;
      const int nr = rows - r0 < kFine ? rows - r0 : kFine;
#pragma unroll
      for (int s = 0; s < S; ++s) h[s] = col ? s_fine[(f * S + s) * D + d] : 0.f;
      for (int q = 0; q < nr; ++q) {
        const int r = r0 + q;
        const float al = s_al[r];
        const float vd = s_v[r * D + d];
#pragma unroll
        for (int s = 0; s < S; ++s) {
          h[s] = fmaf(al, h[s], s_b[r * S + s] * vd);
          if (col) s_st[(q * S + s) * D + d] = h[s];
        }
      }
      __syncwarp();
      for (int q = nr - 1; q >= 0; --q) {
        const int r = r0 + q;
        const int64_t t = t0 + r;
        const float an = s_al[r + 1];  // alpha_{t+1}; 0 past the end
        const float dod = col ? s_do[r * D + d] : 0.f;
        const float vd = col ? s_v[r * D + d] : 0.f;
        // dh_t = c_t do_t^T + alpha_{t+1} dh_{t+1}
#pragma unroll
        for (int s = 0; s < S; ++s) dh[s] = col ? fmaf(an, dh[s], s_c[r * S + s] * dod) : 0.f;
        // dv_t = dh_t^T b_t; dalpha_t = <dh_t, h_{t-1}>
        float dvd = 0.f, dal = 0.f, xb[32], xc[32];
#pragma unroll
        for (int s = 0; s < S; ++s) {
          const float hp = q > 0 ? s_st[((q - 1) * S + s) * D + d] : s_fine[(f * S + s) * D + d];
          const float ht = s_st[(q * S + s) * D + d];
          dvd = fmaf(s_b[r * S + s], dh[s], dvd);
          dal = fmaf(dh[s], col ? hp : 0.f, dal);
          xb[s] = dh[s] * vd;             // db_t[s] = sum_d dh[s][d] v[d]
          xc[s] = col ? ht * dod : 0.f;   // dc_t[s] = sum_d h_t[s][d] do[d]
        }
#pragma unroll
        for (int s = S; s < 32; ++s) {
          xb[s] = 0.f;
          xc[s] = 0.f;
        }
        const float dbs = reduce_scatter32(xb, lane);
        const float dcs = reduce_scatter32(xc, lane);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) dal += __shfl_xor_sync(kFullMask, dal, m);
        if (col) __stcs(p.dv + (bh * T + t) * D + d, dvd);
        if (lane < S) {
          __stcs(p.db + (bh * T + t) * S + lane, dbs);
          __stcs(p.dc + (bh * T + t) * S + lane, dcs);
        }
        if (lane == 0) __stcs(p.dalpha + bh * T + t, dal);
      }
      __syncwarp();
    }
    __syncwarp();
  }
  // dh0 = alpha_0 dh_0
  if (p.dh0 && col && T > 0) {
    const float a0 = __ldg(p.alpha + bh * T);
#pragma unroll
    for (int s = 0; s < S; ++s) p.dh0[(bh * S + s) * D + d] = a0 * dh[s];
  }
}

template <int S, int D>
size_t bwd_smem() {
  return sizeof(float) * ((size_t)kCoarse * (2 * S + 2 * D) + kCoarse + 4 + 4 * S * D +
                          (size_t)kFine * S * D);
}

template <int S, int D>
cudaError_t launch(const GdnParams& p, bool fwd, cudaStream_t s) {
  if (p.BH <= 0 || p.T <= 0) return cudaSuccess;
  if (fwd) {
    gdn_fwd_kernel<S, D><<<(unsigned)p.BH, 32, 0, s>>>(p);
    return cudaGetLastError();
  }
  const size_t smem = bwd_smem<S, D>();
  cudaError_t e = cudaFuncSetAttribute(gdn_bwd_kernel<S, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gdn_bwd_kernel<S, D><<<(unsigned)p.BH, 32, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t dispatch(const GdnParams& p, int S, int D, bool fwd, cudaStream_t s) {
  if (S == 16 && D == 16) return launch<16, 16>(p, fwd, s);
  if (S == 16 && D == 32) return launch<16, 32>(p, fwd, s);
  if (S == 32 && D == 16) return launch<32, 16>(p, fwd, s);
  if (S == 32 && D == 32) return launch<32, 32>(p, fwd, s);
  return cudaErrorInvalidValue;
}

bool shape_ok(int64_t S, int64_t D) { return (S == 16 || S == 32) && (D == 16 || D == 32); }
bool al16(const void* q) { return q == nullptr || ((uintptr_t)q % 16) == 0; }

}  // namespace
}  // namespace scan

using namespace scan;

extern "C" {

size_t gdn_checkpoint_bytes(int64_t B, int64_t H, int64_t T, int64_t S, int64_t D) {
  if (B < 0 || H < 0 || T < 0 || !shape_ok(S, D)) return 0;
  return sizeof(float) * (size_t)(B * H) * (size_t)((T + kCoarse - 1) / kCoarse) * (size_t)(S * D);
}

scan_status gdn_fwd(const float* alpha, const float* b, const float* v, const float* c,
                    const float* h0, float* o, float* ckpt, int64_t B, int64_t H, int64_t T,
                    int64_t S, int64_t D, cudaStream_t stream) {
  if (B < 0 || H < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (!shape_ok(S, D)) return SCAN_ERR_UNSUPPORTED;
  if (B * H * T == 0) return SCAN_OK;
  if (!alpha || !b || !v || !c || !o) return SCAN_ERR_INVALID_ARG;
  if (!al16(b) || !al16(v) || !al16(c) || !al16(h0) || !al16(o) || !al16(ckpt))
    return SCAN_ERR_ALIGNMENT;
  if (B * H > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;
  GdnParams p{};
  p.alpha = alpha;
  p.b = b;
  p.v = v;
  p.c = c;
  p.h0 = h0;
  p.o = o;
  p.ckpt = ckpt;
  p.BH = B * H;
  p.T = T;
  p.NC = (T + kCoarse - 1) / kCoarse;
  return dispatch(p, (int)S, (int)D, true, stream) == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}

scan_status gdn_bwd(const float* alpha, const float* b, const float* v, const float* c,
                    const float* ckpt, const float* dout, float* dalpha, float* db, float* dv,
                    float* dc, float* dh0, int64_t B, int64_t H, int64_t T, int64_t S,
                    int64_t D, cudaStream_t stream) {
  if (B < 0 || H < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (!shape_ok(S, D)) return SCAN_ERR_UNSUPPORTED;
  if (B * H == 0) return SCAN_OK;
  if (T == 0) {
    if (dh0 && cudaMemsetAsync(dh0, 0, sizeof(float) * (size_t)(B * H * S * D), stream) !=
                   cudaSuccess)
      return SCAN_ERR_CUDA;
    return SCAN_OK;
  }
  if (!alpha || !b || !v || !c || !ckpt || !dout || !dalpha || !db || !dv || !dc)
    return SCAN_ERR_INVALID_ARG;
  if (!al16(b) || !al16(v) || !al16(c) || !al16(ckpt) || !al16(dout) || !al16(db) ||
      !al16(dv) || !al16(dc) || !al16(dh0))
    return SCAN_ERR_ALIGNMENT;
  if (B * H > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;
  GdnParams p{};
  p.alpha = alpha;
  p.b = b;
  p.v = v;
  p.c = c;
  p.ckpt = const_cast<float*>(ckpt);
  p.dout = dout;
  p.dalpha = dalpha;
  p.db = db;
  p.dv = dv;
  p.dc = dc;
  p.dh0 = dh0;
  p.BH = B * H;
  p.T = T;
  p.NC = (T + kCoarse - 1) / kCoarse;
  return dispatch(p, (int)S, (int)D, false, stream) == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}

}  // extern "C"
