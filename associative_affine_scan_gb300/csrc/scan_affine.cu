// scan_affine.cu -- block-matrix affine scan H_t = A_t H_{t-1} + B_t.
//
// "Triton scan kernels", One associative-scan family: A_t is k x k, B_t and
// H_t are k x v, and "apply (A1, B1) then (A2, B2)" = (A2 A1, A2 B1 + B2)
// is associative but not commutative, so every composition below keeps the
// time order. The backward ("Autograd integration and the reversed-scan
// backward") is the same scan run from the end over (A_{t+1}^T, dH_t):
// G_t = A_{t+1}^T G_{t+1} + dH_t, dB_t = G_t, dA_t = G_t H_{t-1}^T,
// dh0 = A_0^T G_0, reading only the forward's inputs and output.
//
// Work decomposition: one (b, n) lane is a state block walking T. A block of
// 128 threads takes 32 consecutive lanes (one per thread of a warp, so each
// warp step reads 32 adjacent k x k blocks = one contiguous run of memory) and
// one chunk of 4 * LS steps, split into 4 sub-chunks (one per warp):
//   pass 1: each thread composes its sub-chunk into a summary (P, Q) in fp32
//           registers (time order kept);
//   warp 0: composes the 4 sub-chunk summaries into the chunk summary,
//           publishes it, obtains the chunk's carry-in by a decoupled
//           look-back over earlier chunks' published summaries (bounded
//           waits), publishes the chunk's inclusive state and hands each
//           sub-chunk its own carry-in through shared memory;
//   pass 3: each thread replays its sub-chunk from its carry-in (the chunk's
//           inputs were read microseconds earlier and are served from L2) and
//           writes the outputs.
// Chunks are taken in ticket order, chunk index major, so the chunks a block
// waits for belong to blocks that are already running or finished.
#include <cuda_runtime.h>

#include "scan_scalar.cuh"

namespace scan {
namespace {

constexpr int kSub = 4;  // sub-chunks (warps) per block

// Steps per load batch: a thread issues the loads of PB consecutive steps
// before composing the first of them (k = v = 4: batches of 2 measured faster
// than 4, whose 128 registers halve the resident warps; one step at a time
// was slower still).
constexpr int affine_batch(int k) { return k <= 2 ? 8 : 2; }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// n floats (n % 4 == 0, 16-byte aligned). keep: leave the lines in L2 for a
// second read; otherwise stream (evict first).
template <int N>
__device__ __forceinline__ void ldv(const float* p, float (&r)[N], bool keep) {
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float4 q = keep ? __ldg(reinterpret_cast<const float4*>(p + i))
                          : __ldcs(reinterpret_cast<const float4*>(p + i));
    r[i] = q.x;
    r[i + 1] = q.y;
    r[i + 2] = q.z;
    r[i + 3] = q.w;
  }
}

template <int N>
__device__ __forceinline__ void ldv_cg(const float* p, float (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float4 q = __ldcg(reinterpret_cast<const float4*>(p + i));
    r[i] = q.x;
    r[i + 1] = q.y;
    r[i + 2] = q.z;
    r[i + 3] = q.w;
  }
}

template <int N>
__device__ __forceinline__ void stv(float* p, const float (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4)
    __stcs(reinterpret_cast<float4*>(p + i), make_float4(r[i], r[i + 1], r[i + 2], r[i + 3]));
}

template <int N>
__device__ __forceinline__ void stv_cg(float* p, const float (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4)
    __stcg(reinterpret_cast<float4*>(p + i), make_float4(r[i], r[i + 1], r[i + 2], r[i + 3]));
}

template <int N>
__device__ __forceinline__ void fill(float (&r)[N], float v) {
#pragma unroll
  for (int i = 0; i < N; ++i) r[i] = v;
}

template <int K>
__device__ __forceinline__ void set_identity(float (&r)[K * K]) {
#pragma unroll
  for (int i = 0; i < K; ++i)
#pragma unroll
    for (int j = 0; j < K; ++j) r[i * K + j] = (i == j) ? 1.f : 0.f;
}

// Y = M X (M k x k row-major, X k x w); Y must not alias X.
template <int K, int W>
__device__ __forceinline__ void mul(const float (&M)[K * K], const float (&X)[K * W],
                                    float (&Y)[K * W]) {
#pragma unroll
  for (int i = 0; i < K; ++i)
#pragma unroll
    for (int j = 0; j < W; ++j) {
      float acc = M[i * K] * X[j];
#pragma unroll
      for (int l = 1; l < K; ++l) acc = fmaf(M[i * K + l], X[l * W + j], acc);
      Y[i * W + j] = acc;
    }
}

template <int N>
__device__ __forceinline__ void copy(const float (&s)[N], float (&d)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) d[i] = s[i];
}

// Record of one (lane, chunk) in the workspace: P (k x k), Q (k x v), the
// inclusive state (k x v), then two epoch-tagged flags (summary, inclusive).
template <int K, int V>
struct RecLayout {
  static constexpr int kP = 0;
  static constexpr int kQ = K * K;
  static constexpr int kH = K * K + K * V;
  static constexpr int kFlags = K * K + 2 * K * V;
  static constexpr int kFloats = ((kFlags + 2) + 3) & ~3;
};

// Column j of a block (k x v, row-major): c[i] = X[i][j].
template <int K, int V>
__device__ __forceinline__ void load_col(const float* X, int j, float (&c)[K], bool keep) {
#pragma unroll
  for (int i = 0; i < K; ++i) c[i] = keep ? __ldg(X + i * V + j) : __ldcs(X + i * V + j);
}

template <int K, int V>
__device__ __forceinline__ void store_col(float* X, int j, const float (&c)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) __stcs(X + i * V + j, c[i]);
}

template <int K, int V>
__device__ __forceinline__ void store_col_cg(float* X, int j, const float (&c)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) __stcg(X + i * V + j, c[i]);
}

// y = M x + d (M k x k row-major, x, d k-vectors); y must not alias x
template <int K>
__device__ __forceinline__ void mv_add(const float (&M)[K * K], const float (&x)[K],
                                       const float (&d)[K], float (&y)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) {
    float acc = d[i];
#pragma unroll
    for (int l = 0; l < K; ++l) acc = fmaf(M[i * K + l], x[l], acc);
    y[i] = acc;
  }
}

// y = M^T x + d
template <int K>
__device__ __forceinline__ void mtv_add(const float (&M)[K * K], const float (&x)[K],
                                        const float (&d)[K], float (&y)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) {
    float acc = d[i];
#pragma unroll
    for (int l = 0; l < K; ++l) acc = fmaf(M[l * K + i], x[l], acc);
    y[i] = acc;
  }
}

// Carry-in column j of chunk k of one lane: walk back over the lane's earlier
// chunks, composing their summaries (later ones applied last) until one has
// published its inclusive state. Bounded by p.wait_limit_ns.
template <int K, int V>
__device__ void lookback_col(const AffineParams& p, const float* lane_recs, int k,
                             uint32_t epoch, bool stalled, unsigned ticket, int64_t lane_id,
                             int j, float (&carry)[K]) {
  using RL = RecLayout<K, V>;
  uint32_t tag_agg = (epoch << 2) | 1u, tag_inc = (epoch << 2) | 2u;
  if (stalled) tag_agg = tag_inc = 0xffffffffu;
  float Pacc[K * K], Qacc[K];
  set_identity<K>(Pacc);
  fill(Qacc, 0.f);
  int pos = k - 1;
  const unsigned long long t_begin = global_ns();
  unsigned backoff = 32;
  while (pos >= 0) {
    const float* r = lane_recs + (int64_t)pos * RL::kFloats;
    const unsigned* flags = reinterpret_cast<const unsigned*>(r + RL::kFlags);
    if (ld_acquire_u32(flags + 1) == tag_inc) {
      float Hc[K];
#pragma unroll
      for (int i = 0; i < K; ++i) Hc[i] = __ldcg(r + RL::kH + i * V + j);
      mv_add<K>(Pacc, Hc, Qacc, carry);
      return;
    }
    if (ld_acquire_u32(flags) == tag_agg) {
      float Pp[K * K], Qp[K], tq[K], tp[K * K];
      ldv_cg(r + RL::kP, Pp);
#pragma unroll
      for (int i = 0; i < K; ++i) Qp[i] = __ldcg(r + RL::kQ + i * V + j);
      mv_add<K>(Pacc, Qp, Qacc, tq);  // the earlier chunk is applied first
      mul<K, K>(Pacc, Pp, tp);
      copy(tq, Qacc);
      copy(tp, Pacc);
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
  // chunk 0 always publishes its inclusive state, so this is reached only
  // after a timeout: continue from a zero state
  copy(Qacc, carry);
}

// D holds this thread's rank-1 part G[:, j] H[:, j]^T of dA (k x k). After the
// exchange over the V threads of the lane (xor partners), slot row 0 of D is
// row j of dA summed over all columns. Indices stay compile-time; the thread's
// column bits only select which half it keeps.
template <int K, int V>
__device__ __forceinline__ void reduce_scatter_rows(float (&D)[K * K], int j) {
#pragma unroll
  for (int m = 1; m < V; m <<= 1) {
    const bool hi = (j & m) != 0;
#pragma unroll
    for (int i = 0; i < K; i += 2 * m) {
#pragma unroll
      for (int l = 0; l < K; ++l) {
        const float lo_v = D[i * K + l], hi_v = D[(i + m) * K + l];
        const float send = hi ? lo_v : hi_v;
        const float keep = hi ? hi_v : lo_v;
        D[i * K + l] = keep + __shfl_xor_sync(kFull, send, m);
      }
    }
  }
}

template <int K, int V, int LS, int MODE>
__global__ void __launch_bounds__(128) affine_kernel(const __grid_constant__ AffineParams p) {
  static_assert(K == V, "one thread per column of P and Q needs k == v");
  constexpr int PB = affine_batch(K);  // steps whose loads are in flight together
  static_assert(LS % PB == 0, "sub-chunks are whole batches");
  constexpr int KK = K * K, KV = K * V, NL = 32 / V;
  using RL = RecLayout<K, V>;
  __shared__ float s_P[kSub][NL][KK];
  __shared__ float s_Q[kSub][NL][KV];
  __shared__ float s_in[kSub][NL][KV];
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
  const int ln = lane / V, j = lane % V;  // lane in block, column
  const bool zero_b = (p.flags & AFF_ZERO_B) != 0, eye_h0 = (p.flags & AFF_EYE_H0) != 0;
  const bool acc_da = (p.flags & AFF_ACC_DA) != 0;

  if ((int64_t)ticket < p.ntiles) {
    const int k = (int)(ticket / (unsigned)p.G);
    const int g = (int)(ticket % (unsigned)p.G);
    const int64_t groups_n = (p.N + NL - 1) / NL;
    const int64_t b = g / groups_n;
    const int64_t n = (g % groups_n) * NL + ln;
    const bool active = n < p.N;
    const int m = (MODE == MODE_FWD) ? k : (p.M - 1 - k);
    const int64_t T = p.T;
    const int64_t t_lo = (int64_t)m * (kSub * LS) + (int64_t)warp * LS;
    const int64_t t_hi = t_lo + LS < T ? t_lo + LS : T;
    const int64_t lane_id = b * p.N + (active ? n : 0);
    const int64_t NN = p.N;
    auto blk = [&](int64_t t) -> int64_t { return (b * T + t) * NN + n; };

    // ---- pass 1: column j of the sub-chunk summary (P, Q) ----
    float Pc[K], Qc[K];
#pragma unroll
    for (int i = 0; i < K; ++i) {
      Pc[i] = (i == j) ? 1.f : 0.f;
      Qc[i] = 0.f;
    }
    // The steps are taken in batches of PB: a batch's loads are all issued
    // before its first step is composed, so a thread keeps PB steps of
    // inputs in flight instead of one.
    if (active && t_lo < t_hi) {
      if (MODE == MODE_FWD) {
        for (int64_t t0 = t_lo; t0 < t_hi; t0 += PB) {
          float Ab[PB][KK], Bb[PB][K];
#pragma unroll
          for (int q = 0; q < PB; ++q)
            if (t0 + q < t_hi) {
              ldv(p.A + blk(t0 + q) * KK, Ab[q], true);
              if (zero_b) fill(Bb[q], 0.f);
              else load_col<K, V>(p.Bm + blk(t0 + q) * KV, j, Bb[q], true);
            }
#pragma unroll
          for (int q = 0; q < PB; ++q)
            if (t0 + q < t_hi) {
              float tq[K], tp[K], z[K];
              fill(z, 0.f);
              mv_add<K>(Ab[q], Qc, Bb[q], tq);
              mv_add<K>(Ab[q], Pc, z, tp);
              copy(tq, Qc);
              copy(tp, Pc);
            }
        }
      } else {
        // G_t = A_{t+1}^T G_{t+1} + dH_t, walking t downwards
        for (int64_t t0 = t_hi - 1; t0 >= t_lo; t0 -= PB) {
          float Ab[PB][KK], Db[PB][K];
#pragma unroll
          for (int q = 0; q < PB; ++q) {
            const int64_t t = t0 - q;
            if (t >= t_lo) {
              if (t + 1 < T) ldv(p.A + blk(t + 1) * KK, Ab[q], true);
              else fill(Ab[q], 0.f);
              load_col<K, V>(p.dH + blk(t) * KV, j, Db[q], true);
            }
          }
#pragma unroll
          for (int q = 0; q < PB; ++q)
            if (t0 - q >= t_lo) {
              float tq[K], tp[K], z[K];
              fill(z, 0.f);
              mtv_add<K>(Ab[q], Qc, Db[q], tq);
              mtv_add<K>(Ab[q], Pc, z, tp);
              copy(tq, Qc);
              copy(tp, Pc);
            }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < K; ++i) {
      s_P[warp][ln][i * K + j] = Pc[i];
      s_Q[warp][ln][i * V + j] = Qc[i];
    }
    __syncthreads();

    // ---- chunk summary, look-back, carry-ins (warp 0: 8 lanes x 4 columns) ----
    if (warp == 0) {
      float* lane_recs = p.recs + lane_id * (int64_t)p.M * RL::kFloats;
      float* rec = lane_recs + (int64_t)k * RL::kFloats;
      unsigned* flags = reinterpret_cast<unsigned*>(rec + RL::kFlags);
      const uint32_t tag_agg = (epoch << 2) | 1u, tag_inc = (epoch << 2) | 2u;
      float carry[K];
      fill(carry, 0.f);
      if (active) {
        if (k == 0) {
          if (MODE == MODE_FWD && eye_h0) {
#pragma unroll
            for (int i = 0; i < K; ++i) carry[i] = (i == j) ? 1.f : 0.f;
          } else if (MODE == MODE_FWD && p.h0) {
            load_col<K, V>(p.h0 + lane_id * KV, j, carry, false);
          }
        } else {
          // column j of the chunk summary, sub-chunks in scan order
          float Pt[K], Qt[K];
#pragma unroll
          for (int i = 0; i < K; ++i) {
            Pt[i] = (i == j) ? 1.f : 0.f;
            Qt[i] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < kSub; ++q) {
            const int s = (MODE == MODE_FWD) ? q : kSub - 1 - q;
            float Ps[KK], Qs[K], tq[K], tp[K], z[K];
#pragma unroll
            for (int i = 0; i < KK; ++i) Ps[i] = s_P[s][ln][i];
#pragma unroll
            for (int i = 0; i < K; ++i) Qs[i] = s_Q[s][ln][i * V + j];
            fill(z, 0.f);
            mv_add<K>(Ps, Qt, Qs, tq);
            mv_add<K>(Ps, Pt, z, tp);
            copy(tq, Qt);
            copy(tp, Pt);
          }
#pragma unroll
          for (int i = 0; i < K; ++i) {
            __stcg(rec + RL::kP + i * K + j, Pt[i]);
            __stcg(rec + RL::kQ + i * V + j, Qt[i]);
          }
          __threadfence();
        }
      }
      __syncwarp();
      if (active && k > 0) {
        if (j == 0) st_release_u32(flags, tag_agg);
        const bool stalled = p.test_stall && lane_id == 0 && k == 1;
        lookback_col<K, V>(p, lane_recs, k, epoch, stalled, ticket, lane_id, j, carry);
      }
      if (active) {
        // carry-in of every sub-chunk, and the chunk's inclusive state
#pragma unroll
        for (int q = 0; q < kSub; ++q) {
          const int s = (MODE == MODE_FWD) ? q : kSub - 1 - q;
#pragma unroll
          for (int i = 0; i < K; ++i) s_in[s][ln][i * V + j] = carry[i];
          float Ps[KK], Qs[K], tq[K];
#pragma unroll
          for (int i = 0; i < KK; ++i) Ps[i] = s_P[s][ln][i];
#pragma unroll
          for (int i = 0; i < K; ++i) Qs[i] = s_Q[s][ln][i * V + j];
          mv_add<K>(Ps, carry, Qs, tq);
          copy(tq, carry);
        }
        store_col_cg<K, V>(rec + RL::kH, j, carry);
        __threadfence();
      }
      __syncwarp();
      if (active && j == 0) st_release_u32(flags + 1, tag_inc);
    }
    __syncthreads();

    // ---- pass 3: replay the sub-chunk from its carry-in ----
    float c[K];
#pragma unroll
    for (int i = 0; i < K; ++i) c[i] = s_in[warp][ln][i * V + j];
    const bool work = active && t_lo < t_hi;
    if (MODE == MODE_FWD) {
      if (work) {
        for (int64_t t0 = t_lo; t0 < t_hi; t0 += PB) {
          float Ab[PB][KK], Bb[PB][K];
#pragma unroll
          for (int q = 0; q < PB; ++q)
            if (t0 + q < t_hi) {
              ldv(p.A + blk(t0 + q) * KK, Ab[q], false);
              if (zero_b) fill(Bb[q], 0.f);
              else load_col<K, V>(p.Bm + blk(t0 + q) * KV, j, Bb[q], false);
            }
#pragma unroll
          for (int q = 0; q < PB; ++q)
            if (t0 + q < t_hi) {
              float h[K];
              mv_add<K>(Ab[q], c, Bb[q], h);
              store_col<K, V>(p.out_H + blk(t0 + q) * KV, j, h);
              copy(h, c);
            }
        }
      }
    } else {
      // every thread of the warp runs the same number of steps so the row
      // exchange of dA stays warp-uniform; idle threads compute on zeros
      const int64_t w_lo = (int64_t)m * (kSub * LS) + (int64_t)warp * LS;
      const int64_t w_hi = w_lo + LS < T ? w_lo + LS : T;
      for (int64_t t0 = w_hi - 1; t0 >= w_lo; t0 -= PB) {
        float Ab[PB][KK], Db[PB][K], Hb[PB][K];
#pragma unroll
        for (int q = 0; q < PB; ++q) {
          const int64_t t = t0 - q;
          if (work && t >= w_lo) {
            if (t + 1 < T) ldv(p.A + blk(t + 1) * KK, Ab[q], false);
            else fill(Ab[q], 0.f);
            load_col<K, V>(p.dH + blk(t) * KV, j, Db[q], false);
            if (t >= 1) load_col<K, V>(p.H + blk(t - 1) * KV, j, Hb[q], false);
            else if (eye_h0) {
#pragma unroll
              for (int i = 0; i < K; ++i) Hb[q][i] = (i == j) ? 1.f : 0.f;
            } else if (p.h0) load_col<K, V>(p.h0 + lane_id * KV, j, Hb[q], false);
            else fill(Hb[q], 0.f);
          } else {
            fill(Ab[q], 0.f);
            fill(Db[q], 0.f);
            fill(Hb[q], 0.f);
          }
        }
#pragma unroll
        for (int q = 0; q < PB; ++q) {
          const int64_t t = t0 - q;
          if (t < w_lo) break;  // warp-uniform: w_lo and t0 are the same for every thread
          float gn[K], D[KK];
          mtv_add<K>(Ab[q], c, Db[q], gn);
          copy(gn, c);
          // dA_t = G_t H_{t-1}^T: this column's rank-1 part, summed across the lane
#pragma unroll
          for (int i = 0; i < K; ++i)
#pragma unroll
            for (int l = 0; l < K; ++l) D[i * K + l] = c[i] * Hb[q][l];
          reduce_scatter_rows<K, V>(D, j);
          if (work) {
            if (p.dB) store_col<K, V>(p.dB + blk(t) * KV, j, c);
            float* row = p.dA + blk(t) * KK + j * K;
            if (acc_da) {
#pragma unroll
              for (int l = 0; l < K; ++l) row[l] += D[l];
            } else {
#pragma unroll
              for (int l = 0; l < K; ++l) __stcs(row + l, D[l]);
            }
            if (t == 0 && p.dh0) {
              float A0[KK], d0[K], z[K];
              ldv(p.A + blk(0) * KK, A0, false);
              fill(z, 0.f);
              mtv_add<K>(A0, c, z, d0);
              store_col<K, V>(p.dh0 + lane_id * KV, j, d0);
            }
          }
        }
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
cudaError_t launch_kv(const AffineParams& p, const AffinePlan& pl, cudaStream_t s) {
  if (p.ntiles <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)p.ntiles;
  switch (pl.Lc / kSub) {
    case 16: affine_kernel<K, V, 16, MODE><<<grid, 128, 0, s>>>(p); break;
    case 32: affine_kernel<K, V, 32, MODE><<<grid, 128, 0, s>>>(p); break;
    case 64: affine_kernel<K, V, 64, MODE><<<grid, 128, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// (4, 4) and (2, 2) run the register kernel above; every other shape of the
// envelope runs the column-thread kernel with streamed A (scan_affine_generic.cuh).
template <int MODE>
cudaError_t launch_affine(const AffineParams& p, const AffinePlan& pl, cudaStream_t s) {
  // the ring kernels cover the plain scan (no coefficient-prefix flags)
  if (pl.variant == VAR_STATIONARY && p.flags == 0) return launch_affine_ring(p, MODE, s);
  if (p.k == 4 && p.v == 4) return launch_kv<4, 4, MODE>(p, pl, s);
  if (p.k == 2 && p.v == 2) return launch_kv<2, 2, MODE>(p, pl, s);
  switch (p.k) {
    case 1: return launch_affine_generic_k1(p, MODE, s);
    case 2: return launch_affine_generic_k2(p, MODE, s);
    case 4: return launch_affine_generic_k4(p, MODE, s);
    case 8: return launch_affine_generic_k8(p, MODE, s);
    case 16:
      return MODE == MODE_FWD ? launch_affine_generic_k16_fwd(p, s)
                              : launch_affine_generic_k16_bwd(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

namespace {
bool envelope(int x) { return x == 1 || x == 2 || x == 4 || x == 8 || x == 16; }
}  // namespace

int affine_record_floats(int k, int v) {
  if (!envelope(k) || !envelope(v)) return 0;
  // P (k x k), Q (k x v), inclusive state (k x v), two flags, padded to 16 bytes
  return ((k * k + 2 * k * v + 2) + 3) & ~3;
}

int affine_sub_chunks() { return kSub; }
int affine_lanes_per_block(int k, int v) { return 32 / (k > v ? k : v); }

cudaError_t launch_affine_fwd(const AffineParams& p, const AffinePlan& pl, cudaStream_t s) {
  return launch_affine<MODE_FWD>(p, pl, s);
}

cudaError_t launch_affine_bwd(const AffineParams& p, const AffinePlan& pl, cudaStream_t s) {
  return launch_affine<MODE_BWD>(p, pl, s);
}

}  // namespace scan
