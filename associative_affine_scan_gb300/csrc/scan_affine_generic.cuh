// scan_affine_generic.cuh -- the block-matrix scan H_t = A_t H_{t-1} + B_t for
// every block shape k, v in {1, 2, 4, 8, 16} ("Triton scan kernels", One
// associative-scan family: matrix_affine_scan over (k, v) blocks; its
// conformance envelope).
//
// Same chunk decomposition as the register kernel (scan_affine.cu): a block of
// 4 warps takes the lanes of a few (b, n) state blocks and one chunk of
// 4 * LS steps, one warp per sub-chunk; pass 1 composes each sub-chunk's map
// (P, Q), warp 0 composes the chunk's map, publishes it, finds its carry-in by
// decoupled look-back and hands each sub-chunk its carry-in; pass 3 replays
// the sub-chunk. What changes with the shape:
//   * a lane (one state block) is served by C = max(k, v) column threads:
//     thread c holds column c of P (c < k) and column c of Q and H (c < v);
//   * A_t (k x k, up to 1 KB) is not held in registers: each thread streams it
//     by rows from L1/L2 (the lane's C threads read the same rows);
//   * the look-back never forms a k x k product: it finds the nearest
//     published inclusive state and applies the later chunks' maps to it,
//     column by column (matrix-vector products only);
//   * the backward's dA_t = G_t H_{t-1}^T is summed over the v columns through
//     shared memory: thread c < k writes row c of dA_t.
#pragma once

#include "scan_scalar.cuh"

namespace scan {
namespace affg {

constexpr int kSub = 4;  // sub-chunks (warps) per block

template <int K, int V>
struct Shape {
  static constexpr int C = K > V ? K : V;  // column threads per lane
  static constexpr int NL = 32 / C;        // lanes per warp
  static constexpr int KK = K * K, KV = K * V;
  // workspace record of one (lane, chunk): P (k x k), Q (k x v), the
  // inclusive state (k x v), two epoch-tagged flags (summary, inclusive)
  static constexpr int kP = 0, kQ = KK, kH = KK + KV, kFlags = KK + 2 * KV;
  static constexpr int kFloats = ((kFlags + 2) + 3) & ~3;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Row i of a k x k matrix in global memory, loaded as float4 where k allows.
template <int K>
__device__ __forceinline__ void ld_row(const float* M, int i, float (&r)[K]) {
  if constexpr (K % 4 == 0) {
#pragma unroll
    for (int l = 0; l < K; l += 4) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(M + i * K + l));
      r[l] = q.x;
      r[l + 1] = q.y;
      r[l + 2] = q.z;
      r[l + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int l = 0; l < K; ++l) r[l] = __ldg(M + i * K + l);
  }
}

// (p, q) <- (M p, M q + d) for one column of P and Q; M k x k in global memory.
template <int K>
__device__ __forceinline__ void step_fwd(const float* M, float (&p)[K], float (&q)[K],
                                         const float (&d)[K]) {
  float np[K], nq[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    float r[K];
    ld_row<K>(M, i, r);
    float ap = 0.f, aq = d[i];
#pragma unroll
    for (int l = 0; l < K; ++l) {
      ap = fmaf(r[l], p[l], ap);
      aq = fmaf(r[l], q[l], aq);
    }
    np[i] = ap;
    nq[i] = aq;
  }
#pragma unroll
  for (int i = 0; i < K; ++i) {
    p[i] = np[i];
    q[i] = nq[i];
  }
}

// (p, q) <- (M^T p, M^T q + d); M read by rows: row l scatters into every i.
template <int K>
__device__ __forceinline__ void step_bwd(const float* M, float (&p)[K], float (&q)[K],
                                         const float (&d)[K]) {
  float np[K], nq[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    np[i] = 0.f;
    nq[i] = d[i];
  }
#pragma unroll
  for (int l = 0; l < K; ++l) {
    float r[K];
    ld_row<K>(M, l, r);
#pragma unroll
    for (int i = 0; i < K; ++i) {
      np[i] = fmaf(r[i], p[l], np[i]);
      nq[i] = fmaf(r[i], q[l], nq[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < K; ++i) {
    p[i] = np[i];
    q[i] = nq[i];
  }
}

// y <- S y + e for a k x k matrix S and k x v matrix E in shared memory
// (row-major), y being column c of the state (e = column c of E).
template <int K, int V>
__device__ __forceinline__ void apply_smem(const float* S, const float* E, int c, float (&y)[K]) {
  float ny[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    float acc = c < V ? E[i * V + (c < V ? c : 0)] : 0.f;
#pragma unroll
    for (int l = 0; l < K; ++l) acc = fmaf(S[i * K + l], y[l], acc);
    ny[i] = acc;
  }
#pragma unroll
  for (int i = 0; i < K; ++i) y[i] = ny[i];
}

// The same with S and E in a workspace record (read through L2).
template <int K, int V>
__device__ __forceinline__ void apply_rec(const float* rec, int c, float (&y)[K]) {
  using SH = Shape<K, V>;
  float ny[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    float acc = c < V ? __ldcg(rec + SH::kQ + i * V + (c < V ? c : 0)) : 0.f;
#pragma unroll
    for (int l = 0; l < K; ++l) acc = fmaf(__ldcg(rec + SH::kP + i * K + l), y[l], acc);
    ny[i] = acc;
  }
#pragma unroll
  for (int i = 0; i < K; ++i) y[i] = ny[i];
}

// Carry-in (column c) of chunk k of one lane: walks back over the lane's
// records to the nearest published inclusive state, waiting (bounded by
// p.wait_limit_ns) on records whose summary is not out yet, then applies the
// summaries of the chunks after it, earliest first.
template <int K, int V>
__device__ void lookback_apply(const AffineParams& p, const float* lane_recs, int k, uint32_t epoch,
                               bool stalled, unsigned ticket, int64_t lane_id, int c,
                               float (&carry)[K]) {
  using SH = Shape<K, V>;
  uint32_t tag_agg = (epoch << 2) | 1u, tag_inc = (epoch << 2) | 2u;
  if (stalled) tag_agg = tag_inc = 0xffffffffu;
  int pos = k - 1;
  bool found = false;
  const unsigned long long t_begin = global_ns();
  unsigned backoff = 32;
  while (pos >= 0) {
    const unsigned* flags = reinterpret_cast<const unsigned*>(lane_recs + (int64_t)pos * SH::kFloats +
                                                              SH::kFlags);
    if (ld_acquire(flags + 1) == tag_inc) {
      found = true;
      break;
    }
    if (ld_acquire(flags) == tag_agg) {
      --pos;
      backoff = 32;
      continue;
    }
    if (global_ns() - t_begin > p.wait_limit_ns) {
      set_status(p.hdr, kStatusTimeout);
      p.hdr->info[0] = ticket;
      p.hdr->info[1] = 0;
      p.hdr->info[2] = (unsigned)lane_id;
      p.hdr->info[3] = (unsigned)k;
      break;
    }
    __nanosleep(backoff);
    backoff = backoff < 1024 ? backoff * 2 : 1024;
  }
  // chunk 0 always publishes its inclusive state, so "not found" means the
  // wait ran out: continue from a zero state
#pragma unroll
  for (int i = 0; i < K; ++i) carry[i] = 0.f;
  if (!found) return;
  const float* inc = lane_recs + (int64_t)pos * SH::kFloats;
  if (c < V) {
#pragma unroll
    for (int i = 0; i < K; ++i) carry[i] = __ldcg(inc + SH::kH + i * V + c);
  }
  for (int q = pos + 1; q < k; ++q) apply_rec<K, V>(lane_recs + (int64_t)q * SH::kFloats, c, carry);
}

// y <- M y + d (one column), M k x k in global memory.
template <int K>
__device__ __forceinline__ void col_fwd(const float* M, float (&y)[K], const float (&d)[K]) {
  float ny[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    float r[K];
    ld_row<K>(M, i, r);
    float acc = d[i];
#pragma unroll
    for (int l = 0; l < K; ++l) acc = fmaf(r[l], y[l], acc);
    ny[i] = acc;
  }
#pragma unroll
  for (int i = 0; i < K; ++i) y[i] = ny[i];
}

// y <- M^T y + d (one column).
template <int K>
__device__ __forceinline__ void col_bwd(const float* M, float (&y)[K], const float (&d)[K]) {
  float ny[K];
#pragma unroll
  for (int i = 0; i < K; ++i) ny[i] = d[i];
#pragma unroll
  for (int l = 0; l < K; ++l) {
    float r[K];
    ld_row<K>(M, l, r);
#pragma unroll
    for (int i = 0; i < K; ++i) ny[i] = fmaf(r[i], y[l], ny[i]);
  }
#pragma unroll
  for (int i = 0; i < K; ++i) y[i] = ny[i];
}

// One column of a k x v block in global memory (zeros for c >= v).
template <int K, int V>
__device__ __forceinline__ void ld_col(const float* X, int c, float (&r)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) r[i] = c < V ? __ldg(X + i * V + (c < V ? c : 0)) : 0.f;
}

template <int K, int V>
__device__ __forceinline__ void st_col(float* X, int c, const float (&r)[K]) {
  if (c >= V) return;
#pragma unroll
  for (int i = 0; i < K; ++i) __stcs(X + i * V + c, r[i]);
}

template <int K, int V, int MODE>
__global__ void __launch_bounds__(128) generic_kernel(const __grid_constant__ AffineParams p) {
  using SH = Shape<K, V>;
  constexpr int C = SH::C, NL = SH::NL, KK = SH::KK, KV = SH::KV;
  __shared__ float s_P[kSub][NL][KK];
  __shared__ float s_Q[kSub][NL][KV];
  __shared__ float s_in[kSub][NL][KV];
  __shared__ float s_G[MODE == MODE_BWD ? kSub : 1][NL][KV];  // backward: G_t, H_{t-1}
  __shared__ float s_H[MODE == MODE_BWD ? kSub : 1][NL][KV];
  __shared__ unsigned s_ticket, s_epoch;

  if (threadIdx.x == 0) {
    const unsigned long long te = atomicAdd(&p.hdr->ticket_epoch, 1ull);
    s_ticket = (unsigned)te;
    s_epoch = (unsigned)(te >> 32);
  }
  __syncthreads();
  const unsigned ticket = s_ticket;
  const uint32_t epoch = s_epoch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ln = lane / C, c = lane % C;  // lane (state block) in the warp, column
  const bool zero_b = (p.flags & AFF_ZERO_B) != 0, eye_h0 = (p.flags & AFF_EYE_H0) != 0;
  const bool acc_da = (p.flags & AFF_ACC_DA) != 0;
  const int LS = p.Lc / kSub;

  if ((int64_t)ticket < p.ntiles) {
    const int k = (int)(ticket / (unsigned)p.G);
    const int g = (int)(ticket % (unsigned)p.G);
    const int64_t groups_n = (p.N + NL - 1) / NL;
    const int64_t b = g / groups_n;
    const int64_t n = (g % groups_n) * NL + ln;
    const bool active = n < p.N && ln < NL;
    const int m = (MODE == MODE_FWD) ? k : (p.M - 1 - k);
    const int64_t T = p.T;
    const int64_t t_lo = (int64_t)m * (kSub * LS) + (int64_t)warp * LS;
    const int64_t t_hi = t_lo + LS < T ? t_lo + LS : T;
    const int64_t lane_id = b * p.N + (active ? n : 0);
    const int64_t NN = p.N;
    auto blk = [&](int64_t t) -> int64_t { return (b * T + t) * NN + (active ? n : 0); };
    const int lns = ln < NL ? ln : 0;  // shared-memory slot (threads past NL lanes idle)

    // two steps per loop trip let the next step's loads rise above this one's
    // arithmetic: faster for k = 2 and k = 16 (forward 7-20 %), slower for
    // k = 1 and k = 8 (5-20 %), measured over the envelope
    constexpr int kStepUnroll = (K == 2 || K == 16) ? 2 : 1;
    // ---- pass 1: column c of the sub-chunk summary (P, Q) ----
    float Pc[K], Qc[K];
#pragma unroll
    for (int i = 0; i < K; ++i) {
      Pc[i] = (i == c) ? 1.f : 0.f;
      Qc[i] = 0.f;
    }
    if (active && t_lo < t_hi) {
      if (MODE == MODE_FWD) {
        #pragma unroll kStepUnroll
        for (int64_t t = t_lo; t < t_hi; ++t) {
          float d[K];
          if (zero_b) {
#pragma unroll
            for (int i = 0; i < K; ++i) d[i] = 0.f;
          } else {
            ld_col<K, V>(p.Bm + blk(t) * KV, c, d);
          }
          step_fwd<K>(p.A + blk(t) * KK, Pc, Qc, d);
        }
      } else {
        // G_t = A_{t+1}^T G_{t+1} + dH_t, walking t downwards
        #pragma unroll kStepUnroll
        for (int64_t t = t_hi - 1; t >= t_lo; --t) {
          float d[K];
          ld_col<K, V>(p.dH + blk(t) * KV, c, d);
          if (t + 1 < T) {
            step_bwd<K>(p.A + blk(t + 1) * KK, Pc, Qc, d);
          } else {  // past the end: A = 0
#pragma unroll
            for (int i = 0; i < K; ++i) {
              Pc[i] = 0.f;
              Qc[i] = d[i];
            }
          }
        }
      }
    }
    if (ln < NL) {
#pragma unroll
      for (int i = 0; i < K; ++i) {
        if (c < K) s_P[warp][lns][i * K + (c < K ? c : 0)] = Pc[i];
        if (c < V) s_Q[warp][lns][i * V + (c < V ? c : 0)] = Qc[i];
      }
    }
    __syncthreads();

    // ---- chunk summary, look-back, carry-ins (warp 0) ----
    if (warp == 0) {
      float* lane_recs = p.recs + lane_id * (int64_t)p.M * SH::kFloats;
      float* rec = lane_recs + (int64_t)k * SH::kFloats;
      unsigned* flags = reinterpret_cast<unsigned*>(rec + SH::kFlags);
      const uint32_t tag_agg = (epoch << 2) | 1u, tag_inc = (epoch << 2) | 2u;
      float carry[K];
#pragma unroll
      for (int i = 0; i < K; ++i) carry[i] = 0.f;
      if (active) {
        if (k == 0) {
          if (MODE == MODE_FWD && eye_h0) {
#pragma unroll
            for (int i = 0; i < K; ++i) carry[i] = (i == c && c < V) ? 1.f : 0.f;
          } else if (MODE == MODE_FWD && p.h0) {
            ld_col<K, V>(p.h0 + lane_id * KV, c, carry);
          }
        } else {
          // column c of the chunk summary, sub-chunks in scan order
          float Pt[K], Qt[K];
#pragma unroll
          for (int i = 0; i < K; ++i) {
            Pt[i] = (i == c) ? 1.f : 0.f;
            Qt[i] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < kSub; ++q) {
            const int s = (MODE == MODE_FWD) ? q : kSub - 1 - q;
            float z[K];
            apply_smem<K, V>(s_P[s][lns], s_Q[s][lns], c, Qt);
            // Pt <- P_s Pt (no injection)
#pragma unroll
            for (int i = 0; i < K; ++i) z[i] = 0.f;
#pragma unroll
            for (int i = 0; i < K; ++i) {
              float acc = 0.f;
#pragma unroll
              for (int l = 0; l < K; ++l) acc = fmaf(s_P[s][lns][i * K + l], Pt[l], acc);
              z[i] = acc;
            }
#pragma unroll
            for (int i = 0; i < K; ++i) Pt[i] = z[i];
          }
#pragma unroll
          for (int i = 0; i < K; ++i) {
            if (c < K) __stcg(rec + SH::kP + i * K + (c < K ? c : 0), Pt[i]);
            if (c < V) __stcg(rec + SH::kQ + i * V + (c < V ? c : 0), Qt[i]);
          }
          __threadfence();
        }
      }
      __syncwarp();
      if (active && k > 0) {
        if (c == 0) st_release(flags, tag_agg);
        const bool stalled = p.test_stall && lane_id == 0 && k == 1;
        lookback_apply<K, V>(p, lane_recs, k, epoch, stalled, ticket, lane_id, c, carry);
      }
      if (active) {
        // carry-in of every sub-chunk, and the chunk's inclusive state
#pragma unroll
        for (int q = 0; q < kSub; ++q) {
          const int s = (MODE == MODE_FWD) ? q : kSub - 1 - q;
          if (c < V) {
#pragma unroll
            for (int i = 0; i < K; ++i) s_in[s][lns][i * V + (c < V ? c : 0)] = carry[i];
          }
          apply_smem<K, V>(s_P[s][lns], s_Q[s][lns], c, carry);
        }
        if (c < V) {
#pragma unroll
          for (int i = 0; i < K; ++i) __stcg(rec + SH::kH + i * V + (c < V ? c : 0), carry[i]);
        }
        __threadfence();
      }
      __syncwarp();
      if (active && c == 0) st_release(flags + 1, tag_inc);
    }
    __syncthreads();

    // ---- pass 3: replay the sub-chunk from its carry-in ----
    float h[K];
#pragma unroll
    for (int i = 0; i < K; ++i) h[i] = c < V ? s_in[warp][lns][i * V + (c < V ? c : 0)] : 0.f;
    const bool work = active && t_lo < t_hi;
    if (MODE == MODE_FWD) {
      if (work && c < V) {
        #pragma unroll kStepUnroll
        for (int64_t t = t_lo; t < t_hi; ++t) {
          float d[K];
          if (zero_b) {
#pragma unroll
            for (int i = 0; i < K; ++i) d[i] = 0.f;
          } else {
            ld_col<K, V>(p.Bm + blk(t) * KV, c, d);
          }
          col_fwd<K>(p.A + blk(t) * KK, h, d);
          st_col<K, V>(p.out_H + blk(t) * KV, c, h);
        }
      }
    } else {
      // every thread of the warp walks the same steps (the dA rows are summed
      // over the warp's column threads through shared memory)
      for (int64_t t = t_hi - 1; t >= t_lo; --t) {
        float hp[K];
#pragma unroll
        for (int i = 0; i < K; ++i) hp[i] = 0.f;
        if (work && c < V) {
          float d[K];
          ld_col<K, V>(p.dH + blk(t) * KV, c, d);
          if (t + 1 < T) {
            col_bwd<K>(p.A + blk(t + 1) * KK, h, d);
          } else {
#pragma unroll
            for (int i = 0; i < K; ++i) h[i] = d[i];
          }
          if (p.dB) st_col<K, V>(p.dB + blk(t) * KV, c, h);
          if (t >= 1) ld_col<K, V>(p.H + blk(t - 1) * KV, c, hp);
          else if (eye_h0) {
#pragma unroll
            for (int i = 0; i < K; ++i) hp[i] = (i == c) ? 1.f : 0.f;
          } else if (p.h0) ld_col<K, V>(p.h0 + lane_id * KV, c, hp);
          if (t == 0 && p.dh0) {
            float d0[K], z[K];
#pragma unroll
            for (int i = 0; i < K; ++i) {
              d0[i] = h[i];
              z[i] = 0.f;
            }
            col_bwd<K>(p.A + blk(0) * KK, d0, z);
            st_col<K, V>(p.dh0 + lane_id * KV, c, d0);
          }
          // dA_t = G_t H_{t-1}^T: this column's share goes to shared memory
#pragma unroll
          for (int i = 0; i < K; ++i) {
            s_G[warp][lns][i * V + c] = h[i];
            s_H[warp][lns][i * V + c] = hp[i];
          }
        }
        __syncwarp();
        if (work && c < K) {
          float row[K];
#pragma unroll
          for (int l = 0; l < K; ++l) {
            float acc = 0.f;
#pragma unroll
            for (int cc = 0; cc < V; ++cc)
              acc = fmaf(s_G[warp][lns][c * V + cc], s_H[warp][lns][l * V + cc], acc);
            row[l] = acc;
          }
          float* dst = p.dA + blk(t) * KK + c * K;
          if (acc_da) {
#pragma unroll
            for (int l = 0; l < K; ++l) dst[l] += row[l];
          } else {
#pragma unroll
            for (int l = 0; l < K; ++l) __stcs(dst + l, row[l]);
          }
        }
        __syncwarp();
      }
    }
  } else if (threadIdx.x == 0) {
    set_status(p.hdr, kStatusWorkspace);
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned d = atomicAdd(&p.hdr->done, 1u);
    if (d == gridDim.x - 1) finish_lookback_launch(p.hdr, p.recs, p.rec_bytes, epoch);
  }
}

template <int K, int V, int MODE>
cudaError_t launch_kv(const AffineParams& p, cudaStream_t s) {
  if (p.ntiles <= 0) return cudaSuccess;
  generic_kernel<K, V, MODE><<<(unsigned)p.ntiles, 128, 0, s>>>(p);
  return cudaGetLastError();
}

template <int K, int MODE>
cudaError_t launch_k(const AffineParams& p, cudaStream_t s) {
  switch (p.v) {
    case 1: return launch_kv<K, 1, MODE>(p, s);
    case 2: return launch_kv<K, 2, MODE>(p, s);
    case 4: return launch_kv<K, 4, MODE>(p, s);
    case 8: return launch_kv<K, 8, MODE>(p, s);
    case 16: return launch_kv<K, 16, MODE>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int K>
cudaError_t launch_k(const AffineParams& p, int mode, cudaStream_t s) {
  return mode == MODE_FWD ? launch_k<K, MODE_FWD>(p, s) : launch_k<K, MODE_BWD>(p, s);
}

}  // namespace affg
}  // namespace scan
