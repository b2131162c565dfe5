// scan_gdn.cu -- the scalar-gated outer-product state ("Operations & Triton
// Kernels" (HyMo), The chunked GDN algorithm; Mathematical Derivation of the
// Reverse-Time Backward Pass):
//   h_t = alpha_t h_{t-1} + b_t v_t^T      (S x D state per (batch, head))
//   o_t = h_t^T c_t                         (D-vector)
// and its reverse-time backward with the states recomputed from checkpoints.
//
// Work decomposition: one block per (batch, head) walks T with the state in
// registers, split by columns over D / CW warps (columns of h evolve
// independently); a lane holds S / RG rows of one column. The per-step inputs
// (b_t, c_t, v_t, alpha_t) are staged in shared memory by asynchronous 16-byte
// copies, 32 steps per stage, two stages in flight. The forward stores the
// state before every 64th step (the checkpoints the backward starts from). The
// backward walks those 64-step blocks from the end: it stages the block's
// inputs, recomputes the block's states forward keeping the one before every
// 8th step, and then, for each 8-step piece from the last, recomputes its
// states into registers and runs the adjoint over them:
// dh_t = c_t do_t^T + alpha_{t+1} dh_{t+1}, dv_t = dh_t^T b_t (a column's
// rows summed by shuffles), db_t = dh_t v_t and dc_t = h_t do_t (a
// reduce-scatter of shuffles over the warp's columns, then a sum over warps in
// shared memory once per piece), dalpha_t = <dh_t, h_{t-1}>.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/libscan.h"
#include "scan_internal.h"

namespace scan {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kStage = 32;  // forward: steps per staged block
constexpr int kCoarse = 64;  // checkpoint interval
constexpr int kFine = 8;     // backward: states recomputed at a time

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

// Thread layout of a head's block: warp w owns columns CW w .. CW w + CW - 1
// of h; lane l holds column CW w + (l % CW) and the RS = S / RG rows of row
// group g = l / CW (RG = 32 / CW row groups). Columns evolve independently,
// so the forward needs no exchange between warps; a column's read-out
// o_t[d] = sum_s c_t[s] h_t[s][d] is summed over its row groups by shuffles.
template <int S, int D, int CW_>
struct Layout {
  static constexpr int CW = CW_;       // columns per warp
  static constexpr int RG = 32 / CW;   // row groups
  static constexpr int RS = S / RG;    // rows per lane
  static constexpr int NW = D / CW;    // warps per head
  static constexpr int NT = 32 * NW;   // threads per block
  static_assert(RS >= 1 && RS <= CW && NW >= 1, "layout");
};

// Asynchronous 16-byte copies of n floats (n % 4 == 0) by the block's threads.
__device__ __forceinline__ void stage_block(float* dst, const float* src, int n, int tid, int nt) {
  for (int i = tid; i < n / 4; i += nt) cp_async16(dst + 4 * i, src + 4 * i);
}

// N consecutive floats of shared memory (16-byte aligned for N % 4 == 0,
// 8-byte aligned for N % 4 == 2).
template <int N>
__device__ __forceinline__ void ld_row(const float* src, float (&x)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 q = *reinterpret_cast<const float4*>(src + i);
      x[i] = q.x;
      x[i + 1] = q.y;
      x[i + 2] = q.z;
      x[i + 3] = q.w;
    }
  } else if constexpr (N % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 q = *reinterpret_cast<const float2*>(src + i);
      x[i] = q.x;
      x[i + 1] = q.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = src[i];
  }
}

template <int S, int D, int CW_>
__global__ void __launch_bounds__(Layout<S, D, CW_>::NT) gdn_fwd_kernel(const GdnParams p) {
  using LY = Layout<S, D, CW_>;
  constexpr int CW = LY::CW, RS = LY::RS, NT = LY::NT;
  __shared__ __align__(16) float s_b[2][kStage * S];
  __shared__ __align__(16) float s_c[2][kStage * S];
  __shared__ __align__(16) float s_v[2][kStage * D];
  __shared__ float s_al[2][kStage];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = warp * CW + lane % CW, g = lane / CW, s0 = g * RS;
  const int64_t bh = blockIdx.x;
  if (bh >= p.BH) return;
  const int64_t T = p.T;
  float h[RS];
#pragma unroll
  for (int i = 0; i < RS; ++i) h[i] = p.h0 ? p.h0[(bh * S + s0 + i) * D + d] : 0.f;

  const float* gb = p.b + bh * T * S;
  const float* gc = p.c + bh * T * S;
  const float* gv = p.v + bh * T * D;
  const int nblk = (int)((T + kStage - 1) / kStage);
  auto issue = [&](int blk) {
    const int64_t t0 = (int64_t)blk * kStage;
    const int rows = (int)(T - t0 < kStage ? T - t0 : kStage);
    const int st = blk & 1;
    stage_block(s_b[st], gb + t0 * S, rows * S, tid, NT);
    stage_block(s_c[st], gc + t0 * S, rows * S, tid, NT);
    stage_block(s_v[st], gv + t0 * D, rows * D, tid, NT);
    cp_async_commit();
    if (tid < rows) s_al[st][tid] = __ldg(p.alpha + bh * T + t0 + tid);
  };
  issue(0);
  for (int blk = 0; blk < nblk; ++blk) {
    if (blk + 1 < nblk) {
      issue(blk + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int st = blk & 1;
    const int64_t t0 = (int64_t)blk * kStage;
    const int rows = (int)(T - t0 < kStage ? T - t0 : kStage);
#pragma unroll 4
    for (int r = 0; r < rows; ++r) {
      const int64_t t = t0 + r;
      if (p.ckpt && (t % kCoarse) == 0) {
        float* ck = p.ckpt + (bh * p.NC + t / kCoarse) * S * D;
#pragma unroll
        for (int i = 0; i < RS; ++i) ck[(s0 + i) * D + d] = h[i];
      }
      const float al = s_al[st][r];
      const float vd = s_v[st][r * D + d];
      float bb[RS], cc[RS];
      ld_row<RS>(s_b[st] + r * S + s0, bb);
      ld_row<RS>(s_c[st] + r * S + s0, cc);
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int i = 0; i < RS; ++i) {
        h[i] = fmaf(al, h[i], bb[i] * vd);
        if (i & 1) acc1 = fmaf(cc[i], h[i], acc1);
        else acc0 = fmaf(cc[i], h[i], acc0);
      }
      float o = acc0 + acc1;
#pragma unroll
      for (int m = CW; m < 32; m <<= 1) o += __shfl_xor_sync(kFullMask, o, m);
      if (g == 0) __stcs(p.o + (bh * T + t) * D + d, o);
    }
    __syncthreads();  // the stage is refilled two blocks later
  }
}

// Sum of RS per-lane values over the CW column lanes of a warp (lane bits
// below CW), scattered by recursive halving: afterwards lane j (j = lane % CW
// < RS) holds the total of value j.
template <int RS, int CW>
__device__ __forceinline__ float reduce_scatter_cols(float (&x)[RS], int lane) {
#pragma unroll
  for (int m = RS / 2; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = hi ? x[i] : x[i + m];
      const float keep = hi ? x[i + m] : x[i];
      x[i] = keep + __shfl_xor_sync(kFullMask, send, m);
    }
  }
  float v = x[0];
#pragma unroll
  for (int m = RS; m < CW; m <<= 1) v += __shfl_xor_sync(kFullMask, v, m);  // remaining column bits
  return v;
}

// Shared memory of the backward, in floats: a 64-step block's inputs, the
// state before each 8-step piece (per thread), and two buffers of per-warp
// partial sums for the 8 steps of a piece.
template <int S, int D, int CW_>
struct BwdSmem {
  using LY = Layout<S, D, CW_>;
  static constexpr int RED = 2 * S + LY::RG;  // db, dc, and dalpha per row group
  static constexpr int b = 0;
  static constexpr int c = b + kCoarse * S;
  static constexpr int v = c + kCoarse * S;
  static constexpr int dout = v + kCoarse * D;
  static constexpr int al = dout + kCoarse * D;        // kCoarse + 4
  static constexpr int fine = al + kCoarse + 4;        // [kCoarse / kFine][RS][NT]
  static constexpr int red = fine + (kCoarse / kFine) * S * D;  // [2][kFine][NW][RED]
  static constexpr int total = red + 2 * kFine * LY::NW * RED;
};

template <int S, int D, int CW_>
__global__ void __launch_bounds__(Layout<S, D, CW_>::NT) gdn_bwd_kernel(const GdnParams p) {
  using LY = Layout<S, D, CW_>;
  using SM = BwdSmem<S, D, CW_>;
  constexpr int CW = LY::CW, RG = LY::RG, RS = LY::RS, NW = LY::NW, NT = LY::NT;
  constexpr int RED = SM::RED;
  extern __shared__ __align__(16) float sm[];
  float* s_b = sm + SM::b;
  float* s_c = sm + SM::c;
  float* s_v = sm + SM::v;
  float* s_do = sm + SM::dout;
  float* s_al = sm + SM::al;  // alpha of the block's steps and of the step after it
  float* s_fine = sm + SM::fine;
  float* s_red = sm + SM::red;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = lane % CW, d = warp * CW + j, g = lane / CW, s0 = g * RS;
  const int64_t bh = blockIdx.x;
  if (bh >= p.BH) return;
  const int64_t T = p.T;

  float dh[RS];
#pragma unroll
  for (int i = 0; i < RS; ++i) dh[i] = 0.f;
  int buf = 0;  // which s_red buffer the current piece writes

  for (int64_t J = p.NC - 1; J >= 0; --J) {
    const int64_t t0 = J * kCoarse;
    const int rows = (int)(T - t0 < kCoarse ? T - t0 : kCoarse);
    __syncthreads();  // the previous block's readers are done with the inputs
    stage_block(s_b, p.b + (bh * T + t0) * S, rows * S, tid, NT);
    stage_block(s_c, p.c + (bh * T + t0) * S, rows * S, tid, NT);
    stage_block(s_v, p.v + (bh * T + t0) * D, rows * D, tid, NT);
    stage_block(s_do, p.dout + (bh * T + t0) * D, rows * D, tid, NT);
    cp_async_commit();
    for (int i = tid; i <= rows; i += NT) {
      const int64_t t = t0 + i;
      s_al[i] = t < T ? __ldg(p.alpha + bh * T + t) : 0.f;  // alpha_{T} = 0 past the end
    }
    float h[RS];
#pragma unroll
    for (int i = 0; i < RS; ++i) h[i] = p.ckpt[(bh * p.NC + J) * S * D + (s0 + i) * D + d];
    cp_async_wait<0>();
    __syncthreads();
    // ---- the state before each 8-step piece (each thread its own entries) ----
    const int npiece = (rows + kFine - 1) / kFine;
    const int last_start = (npiece - 1) * kFine;
    for (int r = 0;; ++r) {
      if (r % kFine == 0) {
#pragma unroll
        for (int i = 0; i < RS; ++i) s_fine[((r / kFine) * RS + i) * NT + tid] = h[i];
      }
      if (r == last_start) break;
      const float al = s_al[r];
      const float vd = s_v[r * D + d];
      float bb[RS];
      ld_row<RS>(s_b + r * S + s0, bb);
#pragma unroll
      for (int i = 0; i < RS; ++i) h[i] = fmaf(al, h[i], bb[i] * vd);
    }
    // ---- pieces from the last: states in registers, adjoint backwards ----
    for (int f = npiece - 1; f >= 0; --f) {
      const int r0 = f * kFine;
      const int nr = rows - r0 < kFine ? rows - r0 : kFine;
      float hs[kFine + 1][RS];  // hs[q] = state before step r0 + q
#pragma unroll
      for (int i = 0; i < RS; ++i) hs[0][i] = s_fine[(f * RS + i) * NT + tid];
#pragma unroll
      for (int q = 0; q < kFine; ++q) {
        if (q < nr) {
          const int r = r0 + q;
          const float al = s_al[r];
          const float vd = s_v[r * D + d];
          float bb[RS];
          ld_row<RS>(s_b + r * S + s0, bb);
#pragma unroll
          for (int i = 0; i < RS; ++i) hs[q + 1][i] = fmaf(al, hs[q][i], bb[i] * vd);
        }
      }
      float* red = s_red + buf * (kFine * NW * RED);
#pragma unroll
      for (int q = kFine - 1; q >= 0; --q) {
        if (q < nr) {
          const int r = r0 + q;
          const int64_t t = t0 + r;
          const float an = s_al[r + 1];  // alpha_{t+1}; 0 past the end
          const float dod = s_do[r * D + d];
          const float vd = s_v[r * D + d];
          float bb[RS], cc[RS], xb[RS], xc[RS];
          ld_row<RS>(s_b + r * S + s0, bb);
          ld_row<RS>(s_c + r * S + s0, cc);
          float dvp = 0.f, dal = 0.f;
#pragma unroll
          for (int i = 0; i < RS; ++i) {
            dh[i] = fmaf(an, dh[i], cc[i] * dod);  // dh_t = c_t do_t^T + alpha_{t+1} dh_{t+1}
            dvp = fmaf(bb[i], dh[i], dvp);         // dv_t[d] = sum_s b_t[s] dh_t[s][d]
            dal = fmaf(dh[i], hs[q][i], dal);      // dalpha_t = <dh_t, h_{t-1}>
            xb[i] = dh[i] * vd;                    // db_t[s] = sum_d dh_t[s][d] v_t[d]
            xc[i] = hs[q + 1][i] * dod;            // dc_t[s] = sum_d h_t[s][d] do_t[d]
          }
#pragma unroll
          for (int m = CW; m < 32; m <<= 1) dvp += __shfl_xor_sync(kFullMask, dvp, m);
          if (g == 0) __stcs(p.dv + (bh * T + t) * D + d, dvp);
#pragma unroll
          for (int m = 1; m < CW; m <<= 1) dal += __shfl_xor_sync(kFullMask, dal, m);
          const float wb = reduce_scatter_cols<RS, CW>(xb, lane);
          const float wc = reduce_scatter_cols<RS, CW>(xc, lane);
          float* rq = red + (q * NW + warp) * RED;
          if (j < RS) {
            rq[s0 + j] = wb;
            rq[S + s0 + j] = wc;
          }
          if (j == 0) rq[2 * S + g] = dal;
        }
      }
      __syncthreads();
      // sums over the warps (and row groups, for dalpha) of the piece's steps
      for (int k = tid; k < nr * (2 * S + 1); k += NT) {
        const int q = k / (2 * S + 1), e = k - q * (2 * S + 1);
        const float* rq = red + q * NW * RED;
        const int64_t t = t0 + r0 + q;
        float acc = 0.f;
        if (e < 2 * S) {
#pragma unroll
          for (int w = 0; w < NW; ++w) acc += rq[w * RED + e];
          if (e < S) __stcs(p.db + (bh * T + t) * S + e, acc);
          else __stcs(p.dc + (bh * T + t) * S + (e - S), acc);
        } else {
#pragma unroll
          for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int gg = 0; gg < RG; ++gg) acc += rq[w * RED + 2 * S + gg];
          __stcs(p.dalpha + bh * T + t, acc);
        }
      }
      buf ^= 1;  // the next piece writes the other buffer; this one's readers
                 // finish before the barrier that ends the next piece
    }
  }
  // dh0 = alpha_0 dh_0
  if (p.dh0 && T > 0) {
    const float a0 = __ldg(p.alpha + bh * T);
#pragma unroll
    for (int i = 0; i < RS; ++i) p.dh0[(bh * S + s0 + i) * D + d] = a0 * dh[i];
  }
}

template <int S, int D, int CW>
cudaError_t launch(const GdnParams& p, bool fwd, cudaStream_t s) {
  if (p.BH <= 0 || p.T <= 0) return cudaSuccess;
  using LY = Layout<S, D, CW>;
  if (fwd) {
    gdn_fwd_kernel<S, D, CW><<<(unsigned)p.BH, LY::NT, 0, s>>>(p);
    return cudaGetLastError();
  }
  const size_t smem = sizeof(float) * (size_t)BwdSmem<S, D, CW>::total;
  cudaError_t e = cudaFuncSetAttribute(gdn_bwd_kernel<S, D, CW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gdn_bwd_kernel<S, D, CW><<<(unsigned)p.BH, LY::NT, smem, s>>>(p);
  return cudaGetLastError();
}

// Eight columns per warp (four row groups): measured faster than four columns
// per warp (eight row groups), whose extra warps cost more in per-lane loads
// and shuffles than they recover in latency hiding.
template <int S, int D>
cudaError_t launch(const GdnParams& p, bool fwd, cudaStream_t s) {
  return launch<S, D, 8>(p, fwd, s);
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
