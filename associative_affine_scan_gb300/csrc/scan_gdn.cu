// scan_gdn.cu -- the scalar-gated outer-product state ("Operations & Triton
// Kernels" (HyMo), The chunked GDN algorithm; Mathematical Derivation of the
// Reverse-Time Backward Pass):
//   h_t = alpha_t h_{t-1} + b_t v_t^T      (S x D state per (batch, head))
//   o_t = h_t^T c_t                         (D-vector)
// and its reverse-time backward, started from the forward's checkpoints.
//
// Work decomposition: both directions are cut into chunks (64 steps forward,
// 32 backward: the checkpoint interval) that run in parallel; only the S x D state between
// chunks (forward) or its adjoint (backward) is carried serially, by a short
// kernel per head (see the section on the chunked form below). Within a chunk
// the forward walks the steps with the state in registers, one warp per chunk
// (a lane per column); the backward forms the chunk's gradients as small
// matrix products in shared memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/libscan.h"
#include "scan_internal.h"

namespace scan {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kStage = 16;  // steps per stage of the two-slot input rings
constexpr int kCoarse = 32;  // checkpoint interval

struct GdnParams {
  const float* alpha;  // [B,H,T]
  const float* b;      // [B,H,T,S]
  const float* v;      // [B,H,T,D]
  const float* c;      // [B,H,T,S]
  const float* h0;     // [B,H,S,D] nullable
  float* o;            // forward output [B,H,T,D]
  float* ckpt;         // [B,H,NCK,S,D], NCK = ceil(T / 32): state before step 32 j
  const float* dout;   // backward
  float* dalpha;
  float* db;
  float* dv;
  float* dc;
  float* dh0;          // nullable
  float* wsS;          // workspace [B,H,NC,S,D]: each chunk's state (adjoint) sum,
                       // then the state before (adjoint after) the chunk
  float* wsG;          // [B,H,NC] gate product of each chunk
  int64_t BH, T;
  int64_t NC;   // chunks per head of this direction's launches
  int64_t NCK;  // checkpoints per head
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

// Two fp32 fused multiply-adds in one packed instruction (sm_100 and later):
// {a.x b.x + c.x, a.y b.y + c.y}, each rounded once, as fmaf would.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long A, B, C, R;
  asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(C) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(R) : "l"(A), "l"(B), "l"(C));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(R));
  return r;
}

// {a.x b.x, a.y b.y} in one packed instruction, each rounded once
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long A, B, R;
  asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(R) : "l"(A), "l"(B));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(R));
  return r;
}

// Thread layout of a forward block (one chunk): warp w owns columns
// CW w .. CW w + CW - 1 of h; lane l holds column CW w + (l % CW) and the
// RS = S / RG rows of row group g = l / CW (RG = 32 / CW row groups). Columns
// evolve independently, so the warps never exchange data; a column's read-out
// o_t[d] = sum_s c_t[s] h_t[s][d] is summed over its row groups by shuffles.
template <int S, int D, int CW_>
struct Layout {
  static constexpr int CW = CW_;       // columns per warp
  static constexpr int RG = 32 / CW;   // row groups
  static constexpr int RS = S / RG;    // rows per lane
  static constexpr int NW = D / CW;    // warps per chunk
  static constexpr int NT = 32 * NW;   // threads per block
  static_assert(RS >= 2 && RS % 2 == 0 && RS <= CW && NW >= 1, "layout");
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

// ---------------------------------------------------------------------------
// Both directions run chunked over T: the forward in 64-step chunks, the
// backward in 32-step chunks (the checkpoint interval; its chunk products grow
// with the square of the chunk length, and at 32 steps four blocks share an
// SM). Per chunk of n steps with gates alpha_0 .. alpha_{n-1}:
//   forward:  H_out = Gamma H_in + U,   U = sum_tau w_tau b_tau v_tau^T,
//             w_tau = alpha_{tau+1} .. alpha_{n-1},  Gamma = alpha_0 .. alpha_{n-1};
//   backward: G_in = Gamma G_out + V,   V = sum_t Gamma_t c_t dout_t^T,
//             Gamma_t = alpha_0 .. alpha_t
// (the page's chunked GDN algorithm: a chunk's effect on the state is one
// scale and one rank-n update). A first launch forms U (or V) and Gamma for
// every chunk in parallel; a second walks each head's chunks in order with
// the S x D state (or adjoint) in registers, leaving in the workspace the
// state before (adjoint after) each chunk; a third runs every chunk in
// parallel from it.
// ---------------------------------------------------------------------------

constexpr int kL = kCoarse;  // steps per backward chunk (the checkpoint interval)
constexpr int kLF = 64;      // steps per forward chunk (a whole number of checkpoint intervals)
constexpr int kRatio = kLF / kL;  // checkpoints per forward chunk
static_assert(kLF % kL == 0 && kLF <= 64, "forward chunk");

// The chunk sums run one warp per chunk; a lane owns TM x TN entries of the
// S x D sum (TM = S / 8 rows, TN = D / 4 columns).
template <int S, int D>
struct SumLayout {
  static constexpr int TM = S / 8, TN = D / 4;
};

constexpr int kEPL = kL / 32;  // gates per lane in the backward's scans over a chunk
static_assert(kL % 32 == 0 && kL <= 64, "chunk length");

// Product scans over a chunk's 32 EPL gates, lane l holding elements
// EPL l .. EPL l + EPL - 1 in v. prefix_prods: pi[i] = the product of the
// elements up to and including the lane's i-th, pe[i] = up to and excluding
// it; returns the product of all. suffix_prods: q[i] = the product of the
// elements after the lane's i-th; returns the product of all.
template <int EPL>
__device__ __forceinline__ float prefix_prods(const float (&v)[EPL], float (&pi)[EPL],
                                              float (&pe)[EPL], int lane) {
  float x = 1.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) x *= v[i];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFullMask, x, o);
    if (lane >= o) x *= y;
  }
  float run = __shfl_up_sync(kFullMask, x, 1);
  if (lane == 0) run = 1.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    pe[i] = run;
    run *= v[i];
    pi[i] = run;
  }
  return __shfl_sync(kFullMask, x, 31);
}

template <int EPL>
__device__ __forceinline__ float suffix_prods(const float (&v)[EPL], float (&q)[EPL], int lane) {
  float x = 1.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) x *= v[i];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_down_sync(kFullMask, x, o);
    if (lane + o < 32) x *= y;
  }
  float run = __shfl_down_sync(kFullMask, x, 1);
  if (lane == 31) run = 1.f;
#pragma unroll
  for (int i = EPL - 1; i >= 0; --i) {
    q[i] = run;
    run *= v[i];
  }
  return __shfl_sync(kFullMask, x, 0);
}

// U (FWD: sum_tau w_tau b_tau v_tau^T) or V (sum_t Gamma_t c_t dout_t^T) of
// one chunk into the workspace, with the chunk's gate product.
template <int S, int D, bool FWD>
__global__ void __launch_bounds__(32) gdn_chunk_sum_kernel(const GdnParams p) {
  constexpr int TM = SumLayout<S, D>::TM, TN = SumLayout<S, D>::TN;
  constexpr int kL = FWD ? kLF : ::scan::kL;  // this direction's chunk
  constexpr int kEPL = kL / 32;
  __shared__ __align__(16) float s_x[2][kStage * S];
  __shared__ __align__(16) float s_y[2][kStage * D];
  __shared__ float s_g[kL];
  const int lane = threadIdx.x;
  const int64_t blk = blockIdx.x, bh = blk / p.NC, k = blk - bh * p.NC;
  const int64_t T = p.T, r0 = bh * T + k * kL;
  const int n = (int)(T - k * kL < kL ? T - k * kL : kL);
  const int nst = (n + kStage - 1) / kStage;
  const float* gx = (FWD ? p.b : p.c) + r0 * S;
  const float* gy = (FWD ? p.v : p.dout) + r0 * D;
  auto issue = [&](int st) {  // stage st into slot st & 1
    const int rows = n - st * kStage < kStage ? n - st * kStage : kStage;
    stage_block(s_x[st & 1], gx + st * kStage * S, rows * S, lane, 32);
    stage_block(s_y[st & 1], gy + st * kStage * D, rows * D, lane, 32);
    cp_async_commit();
  };
  issue(0);
  if (nst > 1) issue(1);
  {  // gates past the chunk's end count as 1
    float av[kEPL], g[kEPL], ge[kEPL], all;
#pragma unroll
    for (int i = 0; i < kEPL; ++i) {
      const int t = kEPL * lane + i;
      av[i] = t < n ? __ldg(p.alpha + r0 + t) : 1.f;
    }
    if constexpr (FWD) all = suffix_prods(av, g, lane);
    else all = prefix_prods(av, g, ge, lane);
#pragma unroll
    for (int i = 0; i < kEPL; ++i) s_g[kEPL * lane + i] = g[i];
    if (lane == 0) p.wsG[blk] = all;
  }
  const int si = lane >> 2, dj = lane & 3;
  float2 acc[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
  for (int stg = 0; stg < nst; ++stg) {
    if (stg + 1 < nst) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncwarp();
    const float* sx = s_x[stg & 1];
    const float* sy = s_y[stg & 1];
    const int rows = n - stg * kStage < kStage ? n - stg * kStage : kStage;
#pragma unroll 2
    for (int r = 0; r < rows; ++r) {
      const float g = s_g[stg * kStage + r];
      const float2 g2 = make_float2(g, g);
      float x[TM];
      if constexpr (TM == 4) {
        const float4 q = *reinterpret_cast<const float4*>(sx + r * S + 4 * si);
        x[0] = q.x;
        x[1] = q.y;
        x[2] = q.z;
        x[3] = q.w;
      } else {
        const float2 q = *reinterpret_cast<const float2*>(sx + r * S + 2 * si);
        x[0] = q.x;
        x[1] = q.y;
      }
      float2 y[TN / 2];
#pragma unroll
      for (int j = 0; j < TN / 4; ++j) {
        const float4 q = *reinterpret_cast<const float4*>(sy + r * D + TN * dj + 4 * j);
        y[2 * j] = fmul2(make_float2(q.x, q.y), g2);
        y[2 * j + 1] = fmul2(make_float2(q.z, q.w), g2);
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = ffma2(make_float2(x[i], x[i]), y[j], acc[i][j]);
    }
    __syncwarp();  // slot stg & 1 is read; refill it with stage stg + 2
    if (stg + 2 < nst) issue(stg + 2);
  }
  float* out = p.wsS + blk * S * D;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN / 4; ++j)
      *reinterpret_cast<float4*>(out + (TM * si + i) * D + TN * dj + 4 * j) =
          make_float4(acc[i][2 * j].x, acc[i][2 * j].y, acc[i][2 * j + 1].x, acc[i][2 * j + 1].y);
}

// One thread per 4 entries of a head's S x D state (FWD, chunks in order from
// h0; also written to the checkpoints) or adjoint (chunks from the last, from
// 0; dh0 at the end). The loads of the next 8 chunks are in flight while the
// current 8 are chained.
template <int S, int D, bool FWD>
__global__ void __launch_bounds__(S * D / 4) gdn_carry_kernel(const GdnParams p) {
  constexpr int Q = S * D / 4, G8 = 8;
  const int tid = threadIdx.x;
  const int64_t bh = blockIdx.x, NC = p.NC;
  float4* ws = reinterpret_cast<float4*>(p.wsS + bh * NC * S * D) + tid;
  float4* ck = p.ckpt ? reinterpret_cast<float4*>(p.ckpt + bh * p.NCK * S * D) + tid : nullptr;
  const float* gam = p.wsG + bh * NC;
  auto chunk = [&](int64_t i) { return FWD ? i : NC - 1 - i; };
  float4 H = make_float4(0.f, 0.f, 0.f, 0.f);
  if (FWD && p.h0) H = reinterpret_cast<const float4*>(p.h0 + bh * S * D)[tid];
  float4 U[G8], Un[G8];
  float g[G8], gn[G8];
#pragma unroll
  for (int j = 0; j < G8; ++j)
    if (j < NC) {
      U[j] = __ldcg(ws + chunk(j) * Q);
      g[j] = __ldcg(gam + chunk(j));
    }
  for (int64_t i0 = 0; i0 < NC; i0 += G8) {
#pragma unroll
    for (int j = 0; j < G8; ++j)
      if (i0 + G8 + j < NC) {
        Un[j] = __ldcg(ws + chunk(i0 + G8 + j) * Q);
        gn[j] = __ldcg(gam + chunk(i0 + G8 + j));
      }
#pragma unroll
    for (int j = 0; j < G8; ++j)
      if (i0 + j < NC) {
        const int64_t c = chunk(i0 + j);
        // state before (adjoint after) chunk c; the forward keeps it in the
        // checkpoints when the caller asked for them, else in the workspace
        if (FWD && ck) ck[c * kRatio * Q] = H;
        else ws[c * Q] = H;
        H = make_float4(fmaf(g[j], H.x, U[j].x), fmaf(g[j], H.y, U[j].y), fmaf(g[j], H.z, U[j].z),
                        fmaf(g[j], H.w, U[j].w));
      }
#pragma unroll
    for (int j = 0; j < G8; ++j) {
      U[j] = Un[j];
      g[j] = gn[j];
    }
  }
  if (!FWD && p.dh0) reinterpret_cast<float4*>(p.dh0 + bh * S * D)[tid] = H;
}

// One 64-step chunk per block, from the state before it (the carry left it in
// the checkpoints, or the workspace when there are none); the walk writes the
// checkpoint in the middle of the chunk.
template <int S, int D, int CW_>
__global__ void __launch_bounds__(Layout<S, D, CW_>::NT) gdn_fwd_kernel(const GdnParams p) {
  using LY = Layout<S, D, CW_>;
  constexpr int CW = LY::CW, RS = LY::RS, NT = LY::NT;
  static_assert(kLF % kStage == 0 && kL % kStage == 0, "whole stages per chunk");
  __shared__ __align__(16) float s_b[2][kStage * S];
  __shared__ __align__(16) float s_c[2][kStage * S];
  __shared__ __align__(16) float s_v[2][kStage * D];
  __shared__ float s_al[2][kStage];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = warp * CW + lane % CW, g = lane / CW, s0 = g * RS;
  const int64_t blk = blockIdx.x, bh = blk / p.NC, k = blk - bh * p.NC;
  const int64_t T = p.T, tc = k * kLF;
  const int n = (int)(T - tc < kLF ? T - tc : kLF);
  const int nst = (n + kStage - 1) / kStage;
  float* ckb = p.ckpt ? p.ckpt + (bh * p.NCK + k * kRatio) * S * D : nullptr;  // this chunk's
  const float* gb = p.b + bh * T * S;
  const float* gc = p.c + bh * T * S;
  const float* gv = p.v + bh * T * D;
  // The chunk's gates, kLF / 32 per lane, are loaded first and written to a
  // stage's slot only after its copies and the state's loads are under way
  // (a load stored straight into shared memory would hold the warp there).
  static_assert(NT == 32 && kStage <= 32 && 32 % kStage == 0, "one warp per chunk");
  constexpr int GPL = kLF / 32;
  float gates[GPL];
#pragma unroll
  for (int i = 0; i < GPL; ++i) {
    const int t = 32 * i + lane;
    gates[i] = t < n ? __ldg(p.alpha + bh * T + tc + t) : 0.f;
  }
  auto put_gates = [&](int st) {  // stage st's kStage gates into slot st & 1
    const int e0 = st * kStage, j = lane - (e0 & 31);
    float gv_ = gates[0];
#pragma unroll
    for (int i = 1; i < GPL; ++i)
      if ((e0 >> 5) == i) gv_ = gates[i];
    if (j >= 0 && j < kStage && e0 + j < n) s_al[st & 1][j] = gv_;
  };
  // stage st of the chunk into slot st & 1 (a ring of two)
  auto issue = [&](int st) {
    const int64_t t0 = tc + st * kStage;
    const int rows = n - st * kStage < kStage ? n - st * kStage : kStage;
    const int q = st & 1;
    stage_block(s_b[q], gb + t0 * S, rows * S, tid, NT);
    stage_block(s_c[q], gc + t0 * S, rows * S, tid, NT);
    stage_block(s_v[q], gv + t0 * D, rows * D, tid, NT);
    cp_async_commit();
  };
  issue(0);
  if (nst > 1) issue(1);
  float h[RS];
  {
    const float* hin = ckb ? ckb : p.wsS + blk * S * D;  // where the carry left it
#pragma unroll
    for (int i = 0; i < RS; ++i) h[i] = __ldcg(hin + (s0 + i) * D + d);
  }
  put_gates(0);
  if (nst > 1) put_gates(1);
  for (int stg = 0; stg < nst; ++stg) {
    if (stg + 1 < nst) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();
    const int st = stg & 1;
    const int64_t t0 = tc + stg * kStage;
    const int rows = n - stg * kStage < kStage ? n - stg * kStage : kStage;
    // the checkpoints inside the chunk (the carry wrote the one at its start)
    if (ckb && stg > 0 && (stg * kStage) % kL == 0) {
      float* cq = ckb + (stg * kStage / kL) * S * D;
#pragma unroll
      for (int i = 0; i < RS; ++i) cq[(s0 + i) * D + d] = h[i];
    }
#pragma unroll 4
    for (int r = 0; r < rows; ++r) {
      const int64_t t = t0 + r;
      const float al = s_al[st][r];
      const float vd = s_v[st][r * D + d];
      float bb[RS], cc[RS];
      ld_row<RS>(s_b[st] + r * S + s0, bb);
      ld_row<RS>(s_c[st] + r * S + s0, cc);
      // h = alpha h + b v (the product rounded, then one fused step) and the
      // read-out's two interleaved partial sums, two rows per instruction
      const float2 al2 = make_float2(al, al), vd2 = make_float2(vd, vd);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < RS; i += 2) {
        const float2 bv = fmul2(make_float2(bb[i], bb[i + 1]), vd2);
        const float2 hp = ffma2(al2, make_float2(h[i], h[i + 1]), bv);
        h[i] = hp.x;
        h[i + 1] = hp.y;
        acc = ffma2(make_float2(cc[i], cc[i + 1]), hp, acc);
      }
      float o = acc.x + acc.y;
#pragma unroll
      for (int m = CW; m < 32; m <<= 1) o += __shfl_xor_sync(kFullMask, o, m);
      if (g == 0) __stcs(p.o + (bh * T + t) * D + d, o);
    }
    __syncthreads();  // slot st is read; refill it with stage stg + 2
    if (stg + 2 < nst) {
      issue(stg + 2);
      put_gates(stg + 2);
    }
  }
}

// ---------------------------------------------------------------------------
// Backward, chunked over T ("Operations & Triton Kernels" (HyMo), The chunked
// GDN algorithm, applied to the reverse-time pass). Within a chunk of n <= 32
// steps starting from H_in (the checkpoint) and with G_out, the adjoint of the
// state after the chunk (gradients from later chunks only):
//   Gamma_t = alpha_0 .. alpha_t,  D[t][tau] = alpha_{tau+1} .. alpha_t (tau <= t)
//   dh_t   = sum_{t' >= t} D[t'][t] c_t' dout_t'^T + D[n-1][t] G_out
//   G_in   = sum_t Gamma_t c_t dout_t^T + Gamma_{n-1} G_out      (adjoint of H_in)
// and, with CB[t][tau] = c_t.b_tau, DoV[t][tau] = dout_t.v_tau, P = D o CB,
// dS = D o DoV (elementwise, zero above the diagonal), w_tau = D[n-1][tau]:
//   db_tau = sum_t dS[t][tau] c_t + w_tau G_out v_tau
//   dv_tau = sum_t P[t][tau] dout_t + w_tau G_out^T b_tau
//   dc_t   = sum_tau dS[t][tau] b_tau + Gamma_t H_in dout_t
//   dalpha_r = <dh_r, h_{r-1}>
//            = sum_{t >= r} D[t][r] (Gamma_{r-1} z_t + Y[t][r])
//              + w_r (Gamma_{r-1} <G_out, H_in> + y_r),
//   z_t = c_t^T H_in dout_t, Y[t][r] = sum_{tau < r} D[r-1][tau] CB[t][tau] DoV[t][tau],
//   y_r = sum_{tau < r} D[r-1][tau] b_tau^T G_out v_tau
// (all products of gates, no division, so a gate of 0 is exact). Three
// launches: (1) per chunk, V = sum_t Gamma_t c_t dout_t^T and Gamma_{n-1};
// (2) per head, G_in = V + Gamma_{n-1} G_out from the last chunk to the first,
// leaving each chunk's G_out in the workspace and dh0 = G_in of chunk 0;
// (3) per chunk, the gradients above as small GEMMs in shared memory.
// ---------------------------------------------------------------------------

// Shared memory of the chunk-gradient kernel, in floats. Rows are padded by 4
// floats (16-byte aligned, conflict-free 16-byte reads of consecutive rows).
template <int S, int D>
struct ChunkSmem {
  static constexpr int SP = S + 4, DP = D + 4, LP = kL + 4;
  static constexpr int b = 0;                  // [kL][SP]
  static constexpr int c = b + kL * SP;        // [kL][SP]
  static constexpr int dout = c + kL * SP;     // [kL][DP]
  static constexpr int r1 = dout + kL * DP;    // v, H_in, G_out, G_out^T; then Y; then dS^T
  static constexpr int v = r1;                 // [kL][DP]
  static constexpr int hin = v + kL * DP;      // [S][DP]
  static constexpr int gout = hin + S * DP;    // [S][DP]
  static constexpr int goutT = gout + S * DP;  // [D][SP]
  static constexpr int dsT = r1;               // [kL][LP]
  static constexpr int y = r1;                 // [kL][LP]
  static constexpr int r1_end = goutT + D * SP > r1 + kL * LP ? goutT + D * SP : r1 + kL * LP;
  static constexpr int cb = r1_end;            // [kL][LP]: CB, then P^T
  static constexpr int dov = cb + kL * LP;     // [kL][LP]: DoV, then dS
  static constexpr int al = dov + kL * LP;     // kL + 4 gates (1 past the chunk's end)
  static constexpr int gam = al + kL + 4;      // Gamma_t
  static constexpr int gm1 = gam + kL;         // Gamma_{t-1}
  static constexpr int wdec = gm1 + kL;        // D[n-1][t]
  static constexpr int z = wdec + kL;
  static constexpr int w = z + kL;
  static constexpr int yv = w + kL;            // kL + 4
  static constexpr int red = yv + kL + 4;      // per-warp partial sums
  static constexpr int qf = red + 12;          // [4][kL]: gate products of each row quarter
  static constexpr int qa = qf + 4 * kL;       // [4][kL]: dalpha partial sums of each quarter
  static constexpr int total = qa + 4 * kL;
};

__device__ __forceinline__ float f4(const float4& q, int i) {
  return i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
}

// acc += the dot product of two 4-vectors, as two interleaved partial sums
__device__ __forceinline__ float2 dot4x2(const float4& a, const float4& b, float2 acc) {
  acc = ffma2(make_float2(a.x, a.y), make_float2(b.x, b.y), acc);
  return ffma2(make_float2(a.z, a.w), make_float2(b.z, b.w), acc);
}

// A warp's block of a kL x kL product C[m][n] = sum_k A[m][k] B[n][k] (both
// operands row-major with K consecutive, row strides ap and bp): rows
// m0 + li + 4 i (i < 4), columns n0 + lj + 8 j (j < NJ), written to out (row
// stride LP).
template <int K, int LP, int NJ>
__device__ __forceinline__ void gemm_nt_block(const float* A, int ap, const float* B, int bp,
                                              int m0, int n0, int li, int lj, float* out) {
  float2 acc[4][NJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NJ; ++j) acc[i][j] = make_float2(0.f, 0.f);
#pragma unroll
  for (int kk = 0; kk < K; kk += 4) {
    float4 a[4], q[NJ];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(A + (m0 + li + 4 * i) * ap + kk);
#pragma unroll
    for (int j = 0; j < NJ; ++j) q[j] = *reinterpret_cast<const float4*>(B + (n0 + lj + 8 * j) * bp + kk);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < NJ; ++j) acc[i][j] = dot4x2(a[i], q[j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NJ; ++j) out[(m0 + li + 4 * i) * LP + n0 + lj + 8 * j] = acc[i][j].x + acc[i][j].y;
}

// Threads of the chunk-gradient kernel: 4 per step of the chunk (16 column
// threads x 4 rows per row tile; kL columns x 4 row quarters in the walk).
constexpr int kBwdThreads = 4 * kL;

template <int S, int D>
__global__ void __launch_bounds__(kBwdThreads, 160 / kL) gdn_bwd_chunk_kernel(const GdnParams p) {
  using SM = ChunkSmem<S, D>;
  constexpr int SP = SM::SP, DP = SM::DP, LP = SM::LP, NT = kBwdThreads;
  constexpr int TNS = S / 16, TND = D / 16;  // output columns per thread
  extern __shared__ __align__(16) float sm[];
  float* sb = sm + SM::b;
  float* sc = sm + SM::c;
  float* sdo = sm + SM::dout;
  float* sv = sm + SM::v;
  float* sh = sm + SM::hin;
  float* sg = sm + SM::gout;
  float* sgT = sm + SM::goutT;
  float* sdsT = sm + SM::dsT;
  float* scb = sm + SM::cb;
  float* spT = sm + SM::cb;  // P^T, written over CB once CB is read
  float* sdv = sm + SM::dov;
  float* sy = sm + SM::y;
  float* sal = sm + SM::al;
  float* sgam = sm + SM::gam;
  float* sgm1 = sm + SM::gm1;
  float* swd = sm + SM::wdec;
  float* sz = sm + SM::z;
  float* sw = sm + SM::w;
  float* syv = sm + SM::yv;
  float* sred = sm + SM::red;
  float* sqf = sm + SM::qf;
  float* sqa = sm + SM::qa;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t blk = blockIdx.x, bh = blk / p.NC, k = blk - bh * p.NC;
  const int64_t T = p.T, r0 = bh * T + k * kL;
  const int n = (int)(T - k * kL < kL ? T - k * kL : kL);

  // ---- inputs of the chunk (rows past n zeroed), H_in and G_out, all by
  // asynchronous copies; then G_out^T and <G_out, H_in> from shared memory.
  // The gates are loaded first and stored last, so their latency passes
  // under the copies' issue. ----
  static_assert(NT >= kL + 4, "one gate per thread");
  const float gate = tid < n ? __ldg(p.alpha + r0 + tid) : 1.f;  // 1 past the chunk's end
  for (int i = tid; i < n * (S / 4); i += NT) {
    const int t = i / (S / 4), q = 4 * (i - t * (S / 4));
    cp_async16(sb + t * SP + q, p.b + (r0 + t) * S + q);
    cp_async16(sc + t * SP + q, p.c + (r0 + t) * S + q);
  }
  for (int i = tid; i < n * (D / 4); i += NT) {
    const int t = i / (D / 4), q = 4 * (i - t * (D / 4));
    cp_async16(sv + t * DP + q, p.v + (r0 + t) * D + q);
    cp_async16(sdo + t * DP + q, p.dout + (r0 + t) * D + q);
  }
  {
    const float* hin = p.ckpt + blk * S * D;
    const float* gout = p.wsS + blk * S * D;
    for (int i = tid; i < S * (D / 4); i += NT) {
      const int s_ = i / (D / 4), q = 4 * (i - s_ * (D / 4));
      cp_async16(sh + s_ * DP + q, hin + s_ * D + q);
      cp_async16(sg + s_ * DP + q, gout + s_ * D + q);
    }
  }
  cp_async_commit();
  for (int i = n * SP + tid; i < kL * SP; i += NT) {
    sb[i] = 0.f;
    sc[i] = 0.f;
  }
  for (int i = n * DP + tid; i < kL * DP; i += NT) {
    sv[i] = 0.f;
    sdo[i] = 0.f;
  }
  if (tid < kL + 4) sal[tid] = gate;
  cp_async_wait<0>();
  __syncthreads();
  {
    float win = 0.f;
    if constexpr (S == 32 && D == 32 && SP == 36 && DP == 36 && NT == 128) {
      // by diagonals: lane l takes row l, column (l + k) mod 32, so the reads
      // (bank 5 l + k) and the transposed writes (bank 5 l + 4 k) are free of
      // bank conflicts; warp w takes the diagonals k = 8 w .. 8 w + 7
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int s_ = lane, d = (lane + 8 * warp + it) & 31;
        const float g = sg[s_ * DP + d];
        sgT[d * SP + s_] = g;
        win = fmaf(sh[s_ * DP + d], g, win);
      }
    } else {
      for (int e = tid; e < S * D; e += NT) {
        const int s_ = e / D, d = e - s_ * D;
        const float g = sg[s_ * DP + d];
        sgT[d * SP + s_] = g;
        win = fmaf(sh[s_ * DP + d], g, win);
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) win += __shfl_xor_sync(kFullMask, win, o);
    if (lane == 0) sred[warp] = win;
  }
  __syncthreads();

  // ---- gate products: Gamma_t, Gamma_{t-1} (warp 0); D[n-1][t] (warp 1) ----
  if (warp < 2) {
    float av[kEPL], g[kEPL], ge[kEPL];
#pragma unroll
    for (int i = 0; i < kEPL; ++i) av[i] = sal[kEPL * lane + i];
    if (warp == 0) {
      prefix_prods(av, g, ge, lane);
#pragma unroll
      for (int i = 0; i < kEPL; ++i) {
        sgam[kEPL * lane + i] = g[i];
        sgm1[kEPL * lane + i] = ge[i];
      }
    } else {
      suffix_prods(av, g, lane);
#pragma unroll
      for (int i = 0; i < kEPL; ++i) swd[kEPL * lane + i] = g[i];
    }
  }

  // ---- HDo = dout H_in^T, Gv = v G_out^T, Gb = b G_out, kept in registers:
  // thread rows 4 ri .. 4 ri + 3, columns cj + 16 j (j < TN) ----
  const int ri = tid >> 4, cj = tid & 15;
  float hdo[4][TNS], gv[4][TNS], gb[4][TND];
  {
    float2 ah[4][TNS], ag[4][TNS], ab[4][TND];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < TNS; ++j) ah[i][j] = ag[i][j] = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < TND; ++j) ab[i][j] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int d = 0; d < D; d += 4) {  // HDo[t][s] = sum_d dout[t][d] H_in[s][d]; Gv likewise
      float4 ad[4], av[4], qh[TNS], qg[TNS];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ad[i] = *reinterpret_cast<const float4*>(sdo + (4 * ri + i) * DP + d);
        av[i] = *reinterpret_cast<const float4*>(sv + (4 * ri + i) * DP + d);
      }
#pragma unroll
      for (int j = 0; j < TNS; ++j) {
        qh[j] = *reinterpret_cast<const float4*>(sh + (cj + 16 * j) * DP + d);
        qg[j] = *reinterpret_cast<const float4*>(sg + (cj + 16 * j) * DP + d);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < TNS; ++j) {
          ah[i][j] = dot4x2(ad[i], qh[j], ah[i][j]);
          ag[i][j] = dot4x2(av[i], qg[j], ag[i][j]);
        }
    }
#pragma unroll
    for (int s0 = 0; s0 < S; s0 += 4) {  // Gb[tau][d] = sum_s b[tau][s] G_out^T[d][s]
      float4 a[4], q[TND];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(sb + (4 * ri + i) * SP + s0);
#pragma unroll
      for (int j = 0; j < TND; ++j) q[j] = *reinterpret_cast<const float4*>(sgT + (cj + 16 * j) * SP + s0);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < TND; ++j) ab[i][j] = dot4x2(a[i], q[j], ab[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < TNS; ++j) {
        hdo[i][j] = ah[i][j].x + ah[i][j].y;
        gv[i][j] = ag[i][j].x + ag[i][j].y;
      }
#pragma unroll
      for (int j = 0; j < TND; ++j) gb[i][j] = ab[i][j].x + ab[i][j].y;
    }
  }
  // z_t = c_t . HDo_t and w_tau = b_tau . Gv_tau, summed over a row's 16 column threads
  {
    float zp[4], wp[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      zp[i] = wp[i] = 0.f;
#pragma unroll
      for (int j = 0; j < TNS; ++j) {
        zp[i] = fmaf(sc[(4 * ri + i) * SP + cj + 16 * j], hdo[i][j], zp[i]);
        wp[i] = fmaf(sb[(4 * ri + i) * SP + cj + 16 * j], gv[i][j], wp[i]);
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        zp[i] += __shfl_xor_sync(kFullMask, zp[i], o);
        wp[i] += __shfl_xor_sync(kFullMask, wp[i], o);
      }
    }
    if (cj == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sz[4 * ri + i] = zp[i];
        sw[4 * ri + i] = wp[i];
      }
    }
  }

  // ---- CB = c b^T and DoV = dout v^T (kL x kL); warp w takes the 16-row,
  // kL/2-column block (w / 2, w % 2), skipped when it lies entirely above the
  // diagonal ----
  {
    constexpr int HW = kL / 2;
    const int bi = warp >> 1, bj = warp & 1;
    if (HW * bj <= 16 * bi + 15) {
      gemm_nt_block<S, LP, HW / 8>(sc, SP, sb, SP, 16 * bi, HW * bj, lane >> 3, lane & 7, scb);
      gemm_nt_block<D, LP, HW / 8>(sdo, DP, sv, DP, 16 * bi, HW * bj, lane >> 3, lane & 7, sdv);
    }
  }
  // the column walk below splits rows into quarters; here each (column, quarter)
  // forms the product of the quarter's gates that enter D (rows t > tau)
  constexpr int kQ = kL / 4;      // rows per quarter
  constexpr int kColW = kL / 32;  // warps per quarter (32 columns each)
  {
    const int tau = 32 * (warp % kColW) + lane, q = warp / kColW, tq = kQ * q;
    float f = 1.f;
#pragma unroll
    for (int i = 0; i < kQ; ++i)
      if (tq + i > tau) f *= sal[tq + i];
    sqf[q * kL + tau] = f;
  }
  __syncthreads();

  // ---- Y[t][r] (row t: an affine scan over r with gates alpha_r) and y_r;
  // lane l holds r = kEPL l .. kEPL l + kEPL - 1; a warp scans 4 rows at a time
  // (independent shuffle chains) ----
  {
    float ar[kEPL];
#pragma unroll
    for (int e = 0; e < kEPL; ++e) ar[e] = sal[kEPL * lane + e];
    constexpr int NWp = NT / 32;
    for (int rb = warp; rb <= kL; rb += 4 * NWp) {
      float A[4], X[4], xs[4][kEPL];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = rb + u * NWp;
        A[u] = 1.f;
        X[u] = 0.f;
#pragma unroll
        for (int e = 0; e < kEPL; ++e) {
          const int r = kEPL * lane + e;
          float xv = 0.f;
          if (row < kL) {
            if (r <= row) xv = scb[row * LP + r] * sdv[row * LP + r];
          } else if (row == kL) {
            xv = sw[r];
          }
          xs[u][e] = xv;
          X[u] = fmaf(ar[e], X[u], xv);  // the lane's run composed: state after it from 0
          A[u] *= ar[e];
        }
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float Ap = __shfl_up_sync(kFullMask, A[u], o), Xp = __shfl_up_sync(kFullMask, X[u], o);
          if (lane >= o) {
            X[u] = fmaf(A[u], Xp, X[u]);
            A[u] *= Ap;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = rb + u * NWp;
        float st = __shfl_up_sync(kFullMask, X[u], 1);
        if (lane == 0) st = 0.f;
        if (row <= kL) {
          float* dst = row < kL ? sy + row * LP : syv;
#pragma unroll
          for (int e = 0; e < kEPL; ++e) {
            dst[kEPL * lane + e] = st;  // the state before element r
            st = fmaf(ar[e], st, xs[u][e]);
          }
        }
      }
    }
  }
  __syncthreads();

  // ---- down each column tau: D[t][tau] for t >= tau; dS in place, dS^T and
  // P^T (zero below their diagonals), dalpha_tau. Warp w takes 32 columns over
  // one row quarter, starting from the product of the earlier quarters' gates. ----
  static_assert(kQ % 4 == 0, "whole 16-byte pieces of the transposed rows");
  {
    const int tau = 32 * (warp % kColW) + lane, q = warp / kColW, tq = kQ * q;
    float dec = 1.f;
    for (int i = 0; i < q; ++i) dec *= sqf[i * kL + tau];
    const float gm = sgm1[tau];
    float acc = 0.f, dst[kQ], pst[kQ];
#pragma unroll
    for (int i = 0; i < kQ; ++i) {
      const int t = tq + i;
      float* pd = sdv + t * LP + tau;
      if (t < tau) {
        *pd = 0.f;
        dst[i] = pst[i] = 0.f;
      } else {
        if (t > tau) dec *= sal[t];
        const float ds = dec * *pd;
        pst[i] = dec * scb[t * LP + tau];
        *pd = ds;
        dst[i] = ds;
        acc = fmaf(dec, fmaf(gm, sz[t], sy[t * LP + tau]), acc);
      }
    }
    sqa[q * kL + tau] = acc;
    __syncthreads();  // every read of Y and CB is done: dS^T and P^T take their places
#pragma unroll
    for (int i = 0; i < kQ; i += 4) {
      *reinterpret_cast<float4*>(sdsT + tau * LP + tq + i) =
          make_float4(dst[i], dst[i + 1], dst[i + 2], dst[i + 3]);
      *reinterpret_cast<float4*>(spT + tau * LP + tq + i) =
          make_float4(pst[i], pst[i + 1], pst[i + 2], pst[i + 3]);
    }
  }
  __syncthreads();
  if (tid < kL) {
    const int tau = tid;
    float wtot = 0.f;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) wtot += sred[i];
    const float acc = (sqa[tau] + sqa[kL + tau]) + (sqa[2 * kL + tau] + sqa[3 * kL + tau]);
    if (tau < n) p.dalpha[r0 + tau] = fmaf(swd[tau], fmaf(sgm1[tau], wtot, syv[tau]), acc);
  }

  // ---- db = dS^T c + w o Gv, dv = P^T dout + w o Gb, dc = dS b + Gamma o HDo.
  // The sums run over t (db, dv) and tau (dc) four at a time, two terms per
  // packed instruction: the rows of dS^T, P^T and dS give the pairs (16-byte
  // reads), the columns of c, dout and b two single reads each. ----
  {
    float2 adb[4][TNS], adv[4][TND];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float wd = swd[4 * ri + i];
#pragma unroll
      for (int j = 0; j < TNS; ++j) adb[i][j] = make_float2(wd * gv[i][j], 0.f);
#pragma unroll
      for (int j = 0; j < TND; ++j) adv[i][j] = make_float2(wd * gb[i][j], 0.f);
    }
    // the warp's rows tau are 8 w .. 8 w + 7, and dS^T[tau][t], P^T[tau][t]
    // vanish for t < tau; rows past n are zero
#pragma unroll 1
    for (int t = 8 * warp; t < n; t += 4) {
      float4 ds[4], pp[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ds[i] = *reinterpret_cast<const float4*>(sdsT + (4 * ri + i) * LP + t);
        pp[i] = *reinterpret_cast<const float4*>(spT + (4 * ri + i) * LP + t);
      }
      float2 c01[TNS], c23[TNS], d01[TND], d23[TND];
#pragma unroll
      for (int j = 0; j < TNS; ++j) {
        const float* q = sc + t * SP + cj + 16 * j;
        c01[j] = make_float2(q[0], q[SP]);
        c23[j] = make_float2(q[2 * SP], q[3 * SP]);
      }
#pragma unroll
      for (int j = 0; j < TND; ++j) {
        const float* q = sdo + t * DP + cj + 16 * j;
        d01[j] = make_float2(q[0], q[DP]);
        d23[j] = make_float2(q[2 * DP], q[3 * DP]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < TNS; ++j) {
          adb[i][j] = ffma2(make_float2(ds[i].x, ds[i].y), c01[j], adb[i][j]);
          adb[i][j] = ffma2(make_float2(ds[i].z, ds[i].w), c23[j], adb[i][j]);
        }
#pragma unroll
        for (int j = 0; j < TND; ++j) {
          adv[i][j] = ffma2(make_float2(pp[i].x, pp[i].y), d01[j], adv[i][j]);
          adv[i][j] = ffma2(make_float2(pp[i].z, pp[i].w), d23[j], adv[i][j]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = 4 * ri + i;
      if (m < n) {
#pragma unroll
        for (int j = 0; j < TNS; ++j) __stcs(p.db + (r0 + m) * S + cj + 16 * j, adb[i][j].x + adb[i][j].y);
#pragma unroll
        for (int j = 0; j < TND; ++j) __stcs(p.dv + (r0 + m) * D + cj + 16 * j, adv[i][j].x + adv[i][j].y);
      }
    }
  }
  {
    float2 adc[4][TNS];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float g = sgam[4 * ri + i];
#pragma unroll
      for (int j = 0; j < TNS; ++j) adc[i][j] = make_float2(g * hdo[i][j], 0.f);
    }
    // dS[t][tau] vanishes for tau > t (the warp's rows t end at 8 w + 7)
    const int thi = 8 * warp + 8 < n ? 8 * warp + 8 : n;
#pragma unroll 1
    for (int tau = 0; tau < thi; tau += 4) {
      float4 a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(sdv + (4 * ri + i) * LP + tau);
      float2 b01[TNS], b23[TNS];
#pragma unroll
      for (int j = 0; j < TNS; ++j) {
        const float* q = sb + tau * SP + cj + 16 * j;
        b01[j] = make_float2(q[0], q[SP]);
        b23[j] = make_float2(q[2 * SP], q[3 * SP]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < TNS; ++j) {
          adc[i][j] = ffma2(make_float2(a[i].x, a[i].y), b01[j], adc[i][j]);
          adc[i][j] = ffma2(make_float2(a[i].z, a[i].w), b23[j], adc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = 4 * ri + i;
      if (m < n) {
#pragma unroll
        for (int j = 0; j < TNS; ++j) __stcs(p.dc + (r0 + m) * S + cj + 16 * j, adc[i][j].x + adc[i][j].y);
      }
    }
  }
}

template <int S, int D, int CW>
cudaError_t launch_fwd(const GdnParams& p, cudaStream_t s) {
  const unsigned nblk = (unsigned)(p.BH * p.NC);
  gdn_chunk_sum_kernel<S, D, true><<<nblk, 32, 0, s>>>(p);
  gdn_carry_kernel<S, D, true><<<(unsigned)p.BH, S * D / 4, 0, s>>>(p);
  gdn_fwd_kernel<S, D, CW><<<nblk, Layout<S, D, CW>::NT, 0, s>>>(p);
  return cudaGetLastError();
}

template <int S, int D>
cudaError_t launch_bwd(const GdnParams& p, cudaStream_t s) {
  const unsigned nblk = (unsigned)(p.BH * p.NC);
  gdn_chunk_sum_kernel<S, D, false><<<nblk, 32, 0, s>>>(p);
  gdn_carry_kernel<S, D, false><<<(unsigned)p.BH, S * D / 4, 0, s>>>(p);
  const size_t smem = sizeof(float) * (size_t)ChunkSmem<S, D>::total;
  cudaError_t e = cudaFuncSetAttribute(gdn_bwd_chunk_kernel<S, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gdn_bwd_chunk_kernel<S, D><<<nblk, kBwdThreads, smem, s>>>(p);
  return cudaGetLastError();
}

// Forward: one warp per chunk holding all D columns (CW = D; lane = column, S
// rows per lane when D = 32): with every chunk running in parallel there are
// warps enough, and the wider the column group the fewer shared-memory reads
// of b_t and c_t per state entry. Measured on 8 x 32 heads x 4096 steps,
// S = D = 32: 8 / 16 / 32 columns per warp 0.315 / 0.278 / 0.272 ms.
template <int S, int D>
cudaError_t launch(const GdnParams& p, bool fwd, cudaStream_t s) {
  if (p.BH <= 0 || p.T <= 0) return cudaSuccess;
  return fwd ? launch_fwd<S, D, D>(p, s) : launch_bwd<S, D>(p, s);
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

size_t gdn_workspace_bytes(int64_t B, int64_t H, int64_t T, int64_t S, int64_t D) {
  if (B < 0 || H < 0 || T < 0 || !shape_ok(S, D)) return 0;
  const size_t chunks = (size_t)(B * H) * (size_t)((T + kL - 1) / kL);
  return sizeof(float) * (chunks * (size_t)(S * D) + round_up(chunks, 4));
}

scan_status gdn_fwd(const float* alpha, const float* b, const float* v, const float* c,
                    const float* h0, float* o, float* ckpt, int64_t B, int64_t H, int64_t T,
                    int64_t S, int64_t D, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream) {
  if (B < 0 || H < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (!shape_ok(S, D)) return SCAN_ERR_UNSUPPORTED;
  if (B * H * T == 0) return SCAN_OK;
  if (!alpha || !b || !v || !c || !o) return SCAN_ERR_INVALID_ARG;
  if (!al16(b) || !al16(v) || !al16(c) || !al16(h0) || !al16(o) || !al16(ckpt))
    return SCAN_ERR_ALIGNMENT;
  const int64_t NC = (T + kL - 1) / kL;
  if (B * H * NC > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;
  if (!workspace || !al16(workspace) || workspace_bytes < gdn_workspace_bytes(B, H, T, S, D))
    return SCAN_ERR_WORKSPACE;
  GdnParams p{};
  p.alpha = alpha;
  p.b = b;
  p.v = v;
  p.c = c;
  p.h0 = h0;
  p.o = o;
  p.ckpt = ckpt;
  p.wsS = static_cast<float*>(workspace);
  p.wsG = p.wsS + (size_t)(B * H * NC) * (size_t)(S * D);
  p.BH = B * H;
  p.T = T;
  p.NC = (T + kLF - 1) / kLF;  // the forward's chunks (the workspace holds NC >= these)
  p.NCK = NC;
  return dispatch(p, (int)S, (int)D, true, stream) == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}

scan_status gdn_bwd(const float* alpha, const float* b, const float* v, const float* c,
                    const float* ckpt, const float* dout, float* dalpha, float* db, float* dv,
                    float* dc, float* dh0, int64_t B, int64_t H, int64_t T, int64_t S,
                    int64_t D, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
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
  const int64_t NC = (T + kL - 1) / kL;
  if (B * H * NC > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;
  if (!workspace || !al16(workspace) || workspace_bytes < gdn_workspace_bytes(B, H, T, S, D))
    return SCAN_ERR_WORKSPACE;
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
  p.wsS = static_cast<float*>(workspace);
  p.wsG = p.wsS + (size_t)(B * H * NC) * (size_t)(S * D);
  p.BH = B * H;
  p.T = T;
  p.NC = NC;
  p.NCK = NC;
  return dispatch(p, (int)S, (int)D, false, stream) == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}

}  // extern "C"
