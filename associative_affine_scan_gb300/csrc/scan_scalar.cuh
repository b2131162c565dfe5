// scan_scalar.cuh -- chunked scan kernels for the scalar and log-space forms.
//
// The recurrence h_t = a_t h_{t-1} + x_t ("associative_scan_triton" README,
// quick start) is an affine map per step; a run of steps composes to one map
// h_out = P h_in + Q ("Our RG-LRU GPU audit", Exact real chunk algebra), and
// "apply (P1, Q1) then (P2, Q2)" = (P2 P1, P2 Q1 + Q2) is associative
// ("Triton scan kernels", One associative-scan family). The log-space form
// carries l = log h with the same algebra in (log-coefficient sum, shifted
// log-sum-exp) form.
//
// Work decomposition (one thread block = R rows x one chunk of L = 128 J
// time steps; one warp per row):
//   * each lane owns a run of V = 4 J consecutive steps, loaded as J aligned
//     4-step groups (128-bit fp32 / 64-bit bf16 accesses);
//   * a lane-serial pass composes the run's map (P, Q), a warp-shuffle
//     inclusive scan of the 32 run maps gives each run its chunk-local
//     prefix, and a second lane-serial pass runs the recurrence itself over
//     the run from its carry-in, all in fp32 registers;
//   * the chunk's carry-in comes either from the registers of the same block
//     (STATIONARY: the block walks its row group's chunks in order) or from a
//     decoupled look-back over the published summaries of earlier chunks
//     (LOOKBACK: chunks are independent blocks taken in ticket order, chunk
//     index major, so earlier chunks always belong to running or finished
//     blocks);
//   * outputs are written with vector streaming stores.
//
// Packed sequences (cu_seqlens) never cut the tiling: the first step of every
// sequence (in scan direction) becomes the constant map (0, a h0 + x), which
// erases everything before it exactly, so nothing leaks across sequences
// ("associative_scan_triton" README, how it works). Steps outside [0, T) are
// the identity map and are not written ("Our RG-LRU GPU audit", partial final
// chunks).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <cstring>
#include <type_traits>

#include "scan_internal.h"

namespace scan {

constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned kStatusTimeout = 6u;  // scan_status values
constexpr unsigned kStatusSeqlens = 7u;
constexpr unsigned kStatusWorkspace = 4u;

// ---------------------------------------------------------------------------
// memory access helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return (uint32_t)__cvta_generic_to_shared(ptr);
}

__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned long long pack_rec(uint32_t tag, float v) {
  return ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
}

__device__ __forceinline__ void set_status(WsHeader* hdr, unsigned code) {
  atomicCAS(&hdr->status, 0u, code);
}

template <typename TA>
struct IO;

// Raw: the packed form of 4 consecutive elements as one vector load returns
// it, unpacked to fp32 only when used (loads issued ahead of their use).
template <>
struct IO<float> {
  using Raw = float4;
  static __device__ __forceinline__ Raw ldraw(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
  }
  static __device__ __forceinline__ void unpack(const Raw& q, float v[4]) {
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  }
  static __device__ __forceinline__ void ld4(const float* p, float v[4]) { unpack(ldraw(p), v); }
  static __device__ __forceinline__ float ld1(const float* p) { return __ldcs(p); }
  static __device__ __forceinline__ void st4(float* p, const float v[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  }
  static __device__ __forceinline__ void st1(float* p, float v) { __stcs(p, v); }
};

template <>
struct IO<__nv_bfloat16> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw ldraw(const __nv_bfloat16* p) {
    return __ldcs(reinterpret_cast<const uint2*>(p));
  }
  static __device__ __forceinline__ void unpack(const Raw& q, float v[4]) {
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xffff0000u);
  }
  static __device__ __forceinline__ void ld4(const __nv_bfloat16* p, float v[4]) {
    unpack(ldraw(p), v);
  }
  static __device__ __forceinline__ float ld1(const __nv_bfloat16* p) {
    const unsigned short u = __ldcs(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(((unsigned)u) << 16);
  }
  static __device__ __forceinline__ unsigned pack2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const unsigned*>(&b);
  }
  static __device__ __forceinline__ void st4(__nv_bfloat16* p, const float v[4]) {
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(pack2(v[0], v[1]), pack2(v[2], v[3])));
  }
  static __device__ __forceinline__ void st1(__nv_bfloat16* p, float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    __stcs(reinterpret_cast<unsigned short*>(p), *reinterpret_cast<const unsigned short*>(&b));
  }
};

// 128-byte swizzle of a tile written by a 2-D tensor copy: the 16-byte unit
// index inside each 128-byte row is XORed with the row index mod 8 (tiles
// start on 1024-byte boundaries, the span of the pattern).
__device__ __forceinline__ uint32_t swz128(uint32_t b) { return b ^ ((b >> 3) & 0x70u); }

// Four consecutive elements at element offset o (a multiple of 4) of a
// swizzled tile.
template <typename TA>
struct TIO;

template <>
struct TIO<float> {
  static __device__ __forceinline__ void ld4(const unsigned char* tile, uint32_t o, float v[4]) {
    const float4 q = *reinterpret_cast<const float4*>(tile + swz128(o * 4u));
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  }
  static __device__ __forceinline__ void st4(unsigned char* tile, uint32_t o, const float v[4]) {
    *reinterpret_cast<float4*>(tile + swz128(o * 4u)) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

template <>
struct TIO<__nv_bfloat16> {
  static __device__ __forceinline__ void ld4(const unsigned char* tile, uint32_t o, float v[4]) {
    const uint2 q = *reinterpret_cast<const uint2*>(tile + swz128(o * 2u));
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xffff0000u);
  }
  static __device__ __forceinline__ void st4(unsigned char* tile, uint32_t o, const float v[4]) {
    *reinterpret_cast<uint2*>(tile + swz128(o * 2u)) =
        make_uint2(IO<__nv_bfloat16>::pack2(v[0], v[1]), IO<__nv_bfloat16>::pack2(v[2], v[3]));
  }
};

// One chunk's tiles in shared memory (stream variant).
struct StageView {
  const unsigned char* in[3];  // swizzled input tiles: a, then x (forward) or h, dh (backward)
  unsigned char* out[2];       // swizzled output tiles: h (forward) or dx, da (backward);
                               // null: outputs go straight to global memory
  int64_t e0;                  // row-relative step at tile offset 0
  int64_t c_hi;                // the tiles hold steps [e0, c_hi)
};

// ---------------------------------------------------------------------------
// the two monoids
// ---------------------------------------------------------------------------

// Linear space: E = the map h -> p h + q.
struct LinOp {
  struct E {
    float p, q;
  };
  static __device__ __forceinline__ E identity() { return {1.f, 0.f}; }
  static __device__ __forceinline__ E make(float a, float x) { return {a, x}; }
  // first step of a sequence: the constant map h -> a h0 + x
  static __device__ __forceinline__ E make_first(float a, float x, const float* h0, int64_t i) {
    return {0.f, fmaf(a, h0 ? h0[i] : 0.f, x)};
  }
  // "apply e1 then e2"
  static __device__ __forceinline__ E compose(const E& e1, const E& e2) {
    return {e2.p * e1.p, fmaf(e2.p, e1.q, e2.q)};
  }
  static __device__ __forceinline__ float initial_carry() { return 0.f; }
  // one step of the recurrence on the carried state, the state a sequence's
  // first step produces, and the state as output
  static __device__ __forceinline__ float step(float h, float a, float x) { return fmaf(a, h, x); }
  static __device__ __forceinline__ float first(float a, float x, const float* h0, int64_t i) {
    return fmaf(a, h0 ? h0[i] : 0.f, x);
  }
  static __device__ __forceinline__ float out(float h) { return h; }
  // the carried state of the second lane pass is h itself
  using PState = float;
  static __device__ __forceinline__ PState enter(const E& ex, float c) { return fmaf(ex.p, c, ex.q); }
  static __device__ __forceinline__ float value(const E& e, float c) { return fmaf(e.p, c, e.q); }
  static __device__ __forceinline__ float carry_after(const E& e, float c) { return fmaf(e.p, c, e.q); }
  static __device__ __forceinline__ bool is_const(const E& e) { return e.p == 0.f; }
  static __device__ __forceinline__ float const_carry(const E& e) { return e.q; }
  static __device__ __forceinline__ E from_inc(float c) { return {0.f, c}; }
  static __device__ __forceinline__ E from_agg(float u, float w) { return {u, w}; }
  static __device__ __forceinline__ void to_agg(const E& e, float& u, float& w) {
    u = e.p;
    w = e.q;
  }
  static __device__ __forceinline__ E shfl(const E& e, int src) {
    return {__shfl_sync(kFull, e.p, src), __shfl_sync(kFull, e.q, src)};
  }
  static __device__ __forceinline__ E shfl_up(const E& e, int d) {
    return {__shfl_up_sync(kFull, e.p, d), __shfl_up_sync(kFull, e.q, d)};
  }
  static __device__ __forceinline__ E shfl_down(const E& e, int d) {
    return {__shfl_down_sync(kFull, e.p, d), __shfl_down_sync(kFull, e.q, d)};
  }
  static __device__ __forceinline__ E shfl_xor(const E& e, int d) {
    return {__shfl_xor_sync(kFull, e.p, d), __shfl_xor_sync(kFull, e.q, d)};
  }
};

// log(exp(u) + exp(w)); -inf is the zero term.
__device__ __forceinline__ float log_add_exp(float u, float w) {
  const float m = fmaxf(u, w);
  if (m == -CUDART_INF_F) return -CUDART_INF_F;
  return m + __logf(1.f + __expf(-fabsf(u - w)));
}

// Log space: E = the map l -> log(exp(l + a) + s exp(m)): a is the running
// log-coefficient sum, (m, s) a max-shifted log-sum-exp accumulator ("Triton
// scan kernels", One associative-scan family, parallel_scan_log).
struct LogOp {
  struct E {
    float a, m, s;
  };
  static __device__ __forceinline__ E identity() { return {0.f, -CUDART_INF_F, 0.f}; }
  static __device__ __forceinline__ E make(float la, float lx) { return {la, lx, 1.f}; }
  static __device__ __forceinline__ E make_first(float la, float lx, const float* lh0, int64_t i) {
    if (!lh0) return {-CUDART_INF_F, lx, 1.f};
    const float u = lh0[i] + la;
    const float m = fmaxf(u, lx);
    if (m == -CUDART_INF_F) return {-CUDART_INF_F, -CUDART_INF_F, 0.f};
    return {-CUDART_INF_F, m, __expf(u - m) + __expf(lx - m)};
  }
  static __device__ __forceinline__ E compose(const E& e1, const E& e2) {
    const float u = e1.m + e2.a;  // e1's accumulated mass carried through e2
    const float d = u - e2.m;     // NaN only when both are -inf
    const bool up = u > e2.m;
    float ex = __expf(-fabsf(d));
    if (d != d) ex = 0.f;
    E r;
    r.a = e1.a + e2.a;
    r.m = up ? u : e2.m;
    r.s = up ? fmaf(e2.s, ex, e1.s) : fmaf(e1.s, ex, e2.s);
    return r;
  }
  static __device__ __forceinline__ float initial_carry() { return -CUDART_INF_F; }
  // The second lane pass carries l_t as a max-shifted pair: l = m + log(s),
  // s >= 1 (or m = -inf). A step folds in exp(log a + l) and exp(log x) with
  // one exponential, the output exp(l) = s exp(m) costs one more; no
  // logarithm is taken along the run.
  struct PState {
    float m, s;
  };
  static __device__ __forceinline__ PState enter(const E& ex, float c) {
    const E e = compose(from_inc(c), ex);
    return {e.m, e.s};
  }
  static __device__ __forceinline__ PState step(const PState& st, float la, float lx) {
    const float u = st.m + la;  // the carried mass, shifted
    const float d = u - lx;     // NaN only when both are -inf
    float ex = __expf(-fabsf(d));
    if (d != d) ex = 0.f;
    const bool up = u > lx;
    return {up ? u : lx, up ? st.s + ex : fmaf(st.s, ex, 1.f)};
  }
  static __device__ __forceinline__ PState first(float la, float lx, const float* lh0, int64_t i) {
    const E e = make_first(la, lx, lh0, i);
    return {e.m, e.s};
  }
  static __device__ __forceinline__ float out(const PState& st) { return st.s * __expf(st.m); }
  // linear-space output exp(l_t) for the carry-in log state c
  static __device__ __forceinline__ float value(const E& e, float c) {
    return __expf(c + e.a) + e.s * __expf(e.m);
  }
  static __device__ __forceinline__ float carry_after(const E& e, float c) {
    return log_add_exp(c + e.a, e.m + __logf(e.s));
  }
  static __device__ __forceinline__ bool is_const(const E& e) { return e.a == -CUDART_INF_F; }
  static __device__ __forceinline__ float const_carry(const E& e) { return e.m + __logf(e.s); }
  static __device__ __forceinline__ E from_inc(float c) { return {-CUDART_INF_F, c, 1.f}; }
  static __device__ __forceinline__ E from_agg(float u, float w) { return {u, w, 1.f}; }
  static __device__ __forceinline__ void to_agg(const E& e, float& u, float& w) {
    u = e.a;
    w = e.m + __logf(e.s);
  }
  static __device__ __forceinline__ E shfl(const E& e, int src) {
    return {__shfl_sync(kFull, e.a, src), __shfl_sync(kFull, e.m, src), __shfl_sync(kFull, e.s, src)};
  }
  static __device__ __forceinline__ E shfl_up(const E& e, int d) {
    return {__shfl_up_sync(kFull, e.a, d), __shfl_up_sync(kFull, e.m, d),
            __shfl_up_sync(kFull, e.s, d)};
  }
  static __device__ __forceinline__ E shfl_down(const E& e, int d) {
    return {__shfl_down_sync(kFull, e.a, d), __shfl_down_sync(kFull, e.m, d),
            __shfl_down_sync(kFull, e.s, d)};
  }
  static __device__ __forceinline__ E shfl_xor(const E& e, int d) {
    return {__shfl_xor_sync(kFull, e.a, d), __shfl_xor_sync(kFull, e.m, d),
            __shfl_xor_sync(kFull, e.s, d)};
  }
};

// ---------------------------------------------------------------------------
// packed-sequence window: which positions start a non-empty sequence
// ---------------------------------------------------------------------------

// Packed-sequence lookup: the n + 1 offsets of cu_seqlens, staged once per
// block in shared memory when they fit (otherwise read through the
// read-only cache).
constexpr int kCuSmem = 4096;

struct SegWin {
  const int32_t* cu;
  int n;
};

// Largest i in [0, n-1] with cu[i] <= t: the non-empty sequence holding step
// t (empty sequences share their offset with the next one, which wins). Every
// probe stays inside [0, n-1], whatever cu holds.
__device__ __forceinline__ int seg_find(const SegWin& w, int64_t t) {
  int lo = 0, hi = w.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)w.cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Moves s forward to the sequence holding t (t at or after sequence s).
__device__ __forceinline__ int seg_advance(const SegWin& w, int s, int64_t t) {
  while (s + 1 < w.n && (int64_t)w.cu[s + 1] <= t) ++s;
  return s;
}

// The sequence holding t, starting from a nearby guess s (the one that held
// the previous chunk's steps): a few steps either way, else a full search.
__device__ __forceinline__ int seg_near(const SegWin& w, int s, int64_t t) {
  if (s < 0 || s >= w.n) return seg_find(w, t);
#pragma unroll 1
  for (int it = 0; it < 8; ++it) {
    if ((int64_t)w.cu[s] > t) {
      if (s == 0) return 0;
      --s;
    } else if (s + 1 < w.n && (int64_t)w.cu[s + 1] <= t) {
      ++s;
    } else {
      return s;
    }
  }
  return seg_find(w, t);
}

// Checks 0 = cu[0] <= ... <= cu[n] = T and writes dh0 = 0 for empty sequences.
// Called by every thread of one block.
template <int MODE>
__device__ inline void check_segments(const ScalarParams& p) {
  const int n = p.n_seqs;
  int bad = 0;
  for (int i = threadIdx.x; i <= n; i += blockDim.x) {
    const int64_t c = p.cu[i];
    if (i == 0 && c != 0) bad = 1;
    if (i == n && c != p.T) bad = 1;
    if (i < n && (int64_t)p.cu[i + 1] < c) bad = 1;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(p.hdr, kStatusSeqlens);
  if (MODE != MODE_FWD) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int b = 0; b < p.nbr; ++b) {
      float* dh0 = p.br[b].dh0;
      if (!dh0) continue;
      for (int i = warp; i < n; i += nw) {
        if (p.cu[i] != p.cu[i + 1]) continue;
        for (int64_t c = lane; c < p.rows; c += 32) dh0[(int64_t)i * p.rows + c] = 0.f;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// decoupled look-back
// ---------------------------------------------------------------------------

// Composition in lane order where a higher lane is earlier in scan order.
template <class Op>
__device__ __forceinline__ typename Op::E warp_reduce_ordered(typename Op::E v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const typename Op::E o = Op::shfl_xor(v, off);
    v = (lane & off) ? Op::compose(v, o) : Op::compose(o, v);
  }
  return v;
}

// Carry-in of chunk k of one row: walks the records of chunks k-1, k-2, ...
// 32 at a time until a terminal one (an inclusive state, or a summary that
// is a constant map) and composes everything after it. Every wait is bounded
// by p.wait_limit_ns; on expiry the sticky status becomes SCAN_ERR_TIMEOUT
// and the initial carry is returned, so the kernel always completes.
template <class Op>
__device__ float lookback(const ScalarParams& p, const unsigned long long* recs_row, int k,
                          uint32_t epoch, int lane, unsigned ticket, int brn, int64_t row) {
  uint32_t tag_agg = (epoch << 2) | 1u, tag_inc = (epoch << 2) | 2u;
  if (p.test_stall && brn == 0 && row == 0 && k == 1) tag_agg = tag_inc = 0xffffffffu;
  typename Op::E acc = Op::identity();
  int pos = k - 1;
  const unsigned long long t_begin = global_ns();
  unsigned backoff = 32;
  while (true) {
    const int idx = pos - lane;
    typename Op::E e = Op::identity();
    int st;  // 0 not ready, 1 summary, 2 terminal
    if (idx >= 0) {
      const unsigned long long w1 = ld_relaxed(recs_row + 2 * idx + 1);
      const uint32_t tg = (uint32_t)(w1 >> 32);
      if (tg == tag_inc) {
        e = Op::from_inc(__uint_as_float((uint32_t)w1));
        st = 2;
      } else if (tg == tag_agg) {
        const unsigned long long w0 = ld_relaxed(recs_row + 2 * idx);
        if ((uint32_t)(w0 >> 32) == tag_agg) {
          e = Op::from_agg(__uint_as_float((uint32_t)w0), __uint_as_float((uint32_t)w1));
          st = Op::is_const(e) ? 2 : 1;
        } else {
          st = 0;
        }
      } else {
        st = 0;
      }
    } else {
      e = Op::from_inc(Op::initial_carry());
      st = 2;
    }
    const unsigned term = __ballot_sync(kFull, st == 2);
    const unsigned wait = __ballot_sync(kFull, st == 0);
    const int f = term ? __ffs(term) - 1 : 32;
    const unsigned below = f >= 32 ? kFull : ((1u << f) - 1u);
    if (wait & below) {
      if (__any_sync(kFull, global_ns() - t_begin > p.wait_limit_ns)) {
        if (lane == 0) {
          set_status(p.hdr, kStatusTimeout);
          p.hdr->info[0] = ticket;
          p.hdr->info[1] = (unsigned)brn;
          p.hdr->info[2] = (unsigned)row;
          p.hdr->info[3] = (unsigned)k;
        }
        return Op::initial_carry();
      }
      __nanosleep(backoff);
      backoff = backoff < 1024 ? backoff * 2 : 1024;
      continue;
    }
    if (lane > f) e = Op::identity();
    const typename Op::E win = warp_reduce_ordered<Op>(e, lane);
    acc = Op::compose(win, acc);
    if (f < 32) break;
    pos -= 32;
  }
  return Op::const_carry(acc);
}

// ---------------------------------------------------------------------------
// chunk carry-in: register carry or decoupled look-back
// ---------------------------------------------------------------------------

// The carry entering chunk k of a row, given the chunk's own map blk.
// Stationary: the running carry, advanced past the chunk. Look-back: the
// chunk publishes its summary (or, for the first chunk or a constant map, its
// inclusive state) before it looks back, then its inclusive state.
template <class Op>
__device__ __forceinline__ float chunk_carry_in(const ScalarParams& p, int brn, int64_t row, int k,
                                                bool stationary, uint32_t epoch, unsigned ticket,
                                                const typename Op::E& blk, float& carry) {
  const int lane = threadIdx.x & 31;
  float c;
  if (stationary) {
    c = carry;
    carry = Op::carry_after(blk, c);
    return c;
  }
  unsigned long long* recs_row = p.recs + ((int64_t)brn * p.rows + row) * (int64_t)p.M * 2;
  unsigned long long* rec = recs_row + 2 * (int64_t)k;
  const uint32_t tag_agg = (epoch << 2) | 1u, tag_inc = (epoch << 2) | 2u;
  if (k == 0) {
    c = Op::initial_carry();
    if (lane == 0) st_relaxed(rec + 1, pack_rec(tag_inc, Op::carry_after(blk, c)));
    return c;
  }
  const bool cst = Op::is_const(blk);
  if (lane == 0) {
    if (cst) {
      st_relaxed(rec + 1, pack_rec(tag_inc, Op::const_carry(blk)));
    } else {
      float u, w;
      Op::to_agg(blk, u, w);
      st_relaxed(rec, pack_rec(tag_agg, u));
      st_relaxed(rec + 1, pack_rec(tag_agg, w));
    }
  }
  c = lookback<Op>(p, recs_row, k, epoch, lane, ticket, brn, row);
  if (!cst && lane == 0) st_relaxed(rec + 1, pack_rec(tag_inc, Op::carry_after(blk, c)));
  return c;
}

// ---------------------------------------------------------------------------
// one chunk, interleaved layout (dense fp32 rows)
// ---------------------------------------------------------------------------

// value at memory position (group start + 4): the next lane's first element,
// the next block's lane 0, or the halo after the chunk
template <int J>
__device__ __forceinline__ float next_in_memory(const float (&V)[J][4], int j, float halo, int lane) {
  const float v = __shfl_down_sync(kFull, V[j][0], 1);
  const float vb = (j + 1 < J) ? __shfl_sync(kFull, V[j + 1 < J ? j + 1 : j][0], 0) : halo;
  return lane == 31 ? vb : v;
}

// value at memory position (group start - 1)
template <int J>
__device__ __forceinline__ float prev_in_memory(const float (&V)[J][4], int j, float halo, int lane) {
  const float v = __shfl_up_sync(kFull, V[j][3], 1);
  const float vb = (j > 0) ? __shfl_sync(kFull, V[j > 0 ? j - 1 : 0][3], 31) : halo;
  return lane == 0 ? vb : v;
}

// Lane l holds the 4-step groups at t0 + 128 j + 4 l (j < J): every warp
// load and store is one fully coalesced 512-byte access, at the price of a
// warp scan per 128-step block (the scan order runs across the lanes, then
// across the blocks). Chosen where memory-pipe wavefronts, not arithmetic,
// bound the kernel: dense fp32 rows of the linear form.
template <class Op, int MODE, bool VEC, int J, typename TA, int S>
__device__ __forceinline__ void chunk_groups(const ScalarParams& p, int brn, int64_t row, int k,
                                             bool stationary, uint32_t epoch, unsigned ticket,
                                             float& carry) {
  using E = typename Op::E;
  constexpr int L = 128 * J;
  constexpr bool BWD = MODE == MODE_BWD;
  const BranchArgs& br = p.br[brn];
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;  // the whole warp leaves together
  const int64_t T = p.T;
  const int m = (S > 0) ? k : (p.M - 1 - k);
  const int shift = VEC ? (int)((row * T) & 3) : 0;
  const int64_t t0 = (int64_t)m * L - shift;
  const int64_t roff = row * T;
  const int64_t tl = t0 + 4 * lane;

  float A[J][4], X[J][4], H[J][4];  // H: backward only
  const TA* a = static_cast<const TA*>(br.a) + roff;
  const TA* x = BWD ? nullptr : static_cast<const TA*>(br.x) + roff;
  const float* h = br.h + roff;
  const float* dh = br.dh + roff;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t t = tl + 128 * j;
    if (VEC && t >= 0 && t + 4 <= T) {
      IO<TA>::ld4(a + t, A[j]);
      if (BWD) {
        IO<float>::ld4(h + t, H[j]);
        IO<float>::ld4(dh + t, X[j]);
      } else {
        IO<TA>::ld4(x + t, X[j]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t tt = t + e;
        const bool v = tt >= 0 && tt < T;
        A[j][e] = v ? IO<TA>::ld1(a + tt) : 0.f;
        if (BWD) {
          H[j][e] = v ? IO<float>::ld1(h + tt) : 0.f;
          X[j][e] = v ? IO<float>::ld1(dh + tt) : 0.f;
        } else {
          X[j][e] = v ? IO<TA>::ld1(x + tt) : 0.f;
        }
      }
    }
  }
  // backward halos: the gate one step after (S = -1) or before (S = +1) the
  // chunk, the state one step before (S = -1) or after (S = +1)
  float halo_a = 0.f, halo_h = 0.f;
  if (BWD) {
    if (lane == 0) {
      const int64_t pa = (S < 0) ? t0 + L : t0 - 1;
      const int64_t ph = (S < 0) ? t0 - 1 : t0 + L;
      if (pa >= 0 && pa < T) halo_a = IO<TA>::ld1(a + pa);
      if (ph >= 0 && ph < T) halo_h = IO<float>::ld1(h + ph);
    }
    halo_a = __shfl_sync(kFull, halo_a, 0);
    halo_h = __shfl_sync(kFull, halo_h, 0);
  }

  // ---- elements (dense rows: the recurrence starts at t = 0 or T - 1) ----
  E el[J][4];
  float HN[J];  // backward: cross-lane neighbour state of each group's edge step
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t t = tl + 128 * j;
    float gate[4] = {0.f, 0.f, 0.f, 0.f};
    if (BWD) {
      if (S < 0) {  // causal recurrence: gate a_{t+1}, state h_{t-1}
        gate[0] = A[j][1];
        gate[1] = A[j][2];
        gate[2] = A[j][3];
        gate[3] = next_in_memory<J>(A, j, halo_a, lane);
        HN[j] = prev_in_memory<J>(H, j, halo_h, lane);
      } else {  // reverse recurrence: gate a_{t-1}, state h_{t+1}
        gate[0] = prev_in_memory<J>(A, j, halo_a, lane);
        gate[1] = A[j][0];
        gate[2] = A[j][1];
        gate[3] = A[j][2];
        HN[j] = next_in_memory<J>(H, j, halo_h, lane);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t tt = t + e;
      E v = Op::identity();
      if (tt >= 0 && tt < T) {
        if (!BWD) {
          v = ((S > 0) ? tt == 0 : tt == T - 1) ? Op::make_first(A[j][e], X[j][e], br.h0, row)
                                                : Op::make(A[j][e], X[j][e]);
        } else {
          // the shifted gate is 0 past the end of the row (scan-first step)
          v = Op::make(((S < 0) ? tt == T - 1 : tt == 0) ? 0.f : gate[e], X[j][e]);
        }
      }
      el[j][e] = v;
    }
  }

  // ---- chunk-local inclusive scan in scan order ----
  E blk = Op::identity();
#pragma unroll
  for (int jj = 0; jj < J; ++jj) {
    const int j = (S > 0) ? jj : (J - 1 - jj);
    E lane_tot;
    if (S > 0) {
#pragma unroll
      for (int e = 1; e < 4; ++e) el[j][e] = Op::compose(el[j][e - 1], el[j][e]);
      lane_tot = el[j][3];
    } else {
#pragma unroll
      for (int e = 2; e >= 0; --e) el[j][e] = Op::compose(el[j][e + 1], el[j][e]);
      lane_tot = el[j][0];
    }
    E inc = lane_tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const E o = (S > 0) ? Op::shfl_up(inc, off) : Op::shfl_down(inc, off);
      const bool has = (S > 0) ? (lane >= off) : (lane + off < 32);
      if (has) inc = Op::compose(o, inc);
    }
    E ex = (S > 0) ? Op::shfl_up(inc, 1) : Op::shfl_down(inc, 1);
    if (lane == ((S > 0) ? 0 : 31)) ex = Op::identity();
    const E pre = Op::compose(blk, ex);
#pragma unroll
    for (int e = 0; e < 4; ++e) el[j][e] = Op::compose(pre, el[j][e]);
    blk = Op::compose(blk, Op::shfl(inc, (S > 0) ? 31 : 0));
  }

  const float c = chunk_carry_in<Op>(p, brn, row, k, stationary, epoch, ticket, blk, carry);

  // ---- outputs ----
  if (!BWD) {
    float* hout = br.out_h + roff;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t t = tl + 128 * j;
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = Op::value(el[j][e], c);
      if (VEC && t >= 0 && t + 4 <= T) {
        IO<float>::st4(hout + t, v);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (t + e >= 0 && t + e < T) IO<float>::st1(hout + t + e, v[e]);
      }
    }
  } else {
    TA* dx = static_cast<TA*>(br.dx) + roff;
    TA* da = static_cast<TA*>(br.da) + roff;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t t = tl + 128 * j;
      float gx[4], ga[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t tt = t + e;
        const float gv = Op::value(el[j][e], c);
        float hn;
        if (S < 0) hn = (e > 0) ? H[j][e > 0 ? e - 1 : 0] : HN[j];
        else hn = (e < 3) ? H[j][e < 3 ? e + 1 : 3] : HN[j];
        // the step that starts the forward recurrence reads h0 and feeds dh0
        if ((S < 0) ? tt == 0 : tt == T - 1) {
          hn = br.h0 ? br.h0[row] : 0.f;
          if (br.dh0) br.dh0[row] = A[j][e] * gv;
        }
        gx[e] = gv;
        ga[e] = gv * hn;
      }
      if (VEC && t >= 0 && t + 4 <= T) {
        IO<TA>::st4(dx + t, gx);
        IO<TA>::st4(da + t, ga);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (t + e >= 0 && t + e < T) {
            IO<TA>::st1(dx + t + e, gx[e]);
            IO<TA>::st1(da + t + e, ga[e]);
          }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// one chunk of one row group
// ---------------------------------------------------------------------------

// Each lane owns a run of V = 4 J consecutive steps of the chunk (lane l:
// steps t0 + V l ... t0 + V l + V - 1), read as J aligned 4-step groups.
// The chunk costs one lane-serial pass to compose the run's map, one warp
// scan over the 32 run maps, and one lane-serial pass that runs the
// recurrence itself from the run's carry-in: about three arithmetic
// instructions per step plus V-amortised shuffles.
//
// S is the scan direction: +1 walks t upwards, -1 downwards. A forward call
// scans in the recurrence's direction; a backward call scans against it.
// SMEM: the chunk's inputs are read from the swizzled tiles of sv where they
// hold them (else from global memory), and its outputs go to sv's output
// tiles when it has them. seg_hint (packed sequences): the sequence that held
// this lane's run in the previous chunk, -1 if none; updated for the next
// chunk. release() is called by every lane once the chunk's inputs are in
// registers (the stream variant refills the stage there).
struct NoRelease {
  __device__ __forceinline__ void operator()() const {}
};

// The register-carry loop's loads one chunk ahead: a lane's vector loads of
// the next chunk of its row (raw, the aligned in-row 4-step groups only) and
// the backward gate halo, issued before the current chunk is computed so that
// each warp keeps two chunks of loads in flight. The backward's states h are
// not among them: they are first used after the scan, so their loads,
// issued at the chunk's start, already overlap it.
template <int J, typename TA, int MODE>
struct RunAhead {
  static constexpr bool BWD = MODE != MODE_FWD;
  static constexpr bool LOGIN = MODE == MODE_LOGBWD;
  using XT = typename std::conditional<BWD, float, TA>::type;
  typename IO<TA>::Raw a[J];
  typename IO<XT>::Raw x[J];  // x forward, dh backward
  float4 lx[LOGIN ? J : 1];
  float halo_a;  // backward: the gate halo
  bool full;     // holds the chunk this call is about to scan
};

// Look-ahead pays where a launch's warps are all resident at once and each
// keeps too few bytes in flight: the packed bf16 forward (one wave of
// row-warps, 2-byte inputs, 8 more registers at 256-step chunks). Elsewhere
// its registers cost more occupancy than it gains; the packed backward,
// which already moves 14 bytes per step, measured slower with it.
template <int MODE, bool VARLEN, typename TA>
__host__ __device__ constexpr bool uses_ahead() {
  return MODE == MODE_FWD && VARLEN && sizeof(TA) == 2;
}

// INSIDE: every 4-step group of every lane lies inside the row (vector path,
// not the stream variant's tiles); the per-group bounds checks fold away, and
// packed rows test once per chunk whether any sequence starts or ends in it.
template <class Op, int MODE, bool VARLEN, bool VEC, int J, typename TA, int S, bool SMEM,
          class Release, bool INSIDE>
__device__ __forceinline__ void chunk_body(const ScalarParams& p, int brn, int64_t row, int k,
                                           bool stationary, uint32_t epoch, unsigned ticket,
                                           const SegWin& win, float& carry, const StageView* sv,
                                           int* seg_hint, const Release& release,
                                           RunAhead<J, TA, MODE>* ahead, bool next) {
  using E = typename Op::E;
  constexpr int L = 128 * J;
  constexpr int V = 4 * J;
  constexpr bool BWD = MODE != MODE_FWD;
  constexpr bool LOGIN = MODE == MODE_LOGBWD;  // backward of the log-space form
  const BranchArgs& br = p.br[brn];
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;  // the whole warp leaves together
  const int64_t T = p.T;
  const int m = (S > 0) ? k : (p.M - 1 - k);
  // rows are cut so that every 4-step group starts on a 4-element boundary of
  // memory (16 bytes fp32, 8 bytes bf16), or for tensor-copied tiles on a
  // 128-byte row of the flat tensor, whatever T is
  constexpr int kAlign = SMEM ? tma_row_elems((int)sizeof(TA)) : 4;
  const int shift = VEC ? (int)((row * T) & (kAlign - 1)) : 0;
  const int64_t t0 = (int64_t)m * L - shift;
  const int64_t roff = row * T;
  const int64_t tr = t0 + (int64_t)V * lane;  // first step of this lane's run

  // ---- loads: A = gates, X = inputs (forward) or dh (backward), H = states,
  // LX = log x (log-space backward) ----
  float A[V], X[V], H[BWD ? V : 1], LX[LOGIN ? V : 1];
  const TA* a = static_cast<const TA*>(br.a) + roff;
  const void* xsrc = BWD ? static_cast<const void*>(br.dh) : br.x;
  using XT = typename RunAhead<J, TA, MODE>::XT;  // element type of xsrc
#pragma unroll
  for (int i = 0; i < J; ++i) {
    const int64_t t = tr + 4 * i;
    float* ai = A + 4 * i;
    float* xi = X + 4 * i;
    float* hi = H + (BWD ? 4 * i : 0);
    const bool g_in = INSIDE || (t >= 0 && t + 4 <= T);  // the group lies in the row
    if (SMEM && t + 4 <= sv->c_hi) {
      const uint32_t o = (uint32_t)(t - sv->e0);
      TIO<TA>::ld4(sv->in[0], o, ai);
      if (BWD) {
        TIO<float>::ld4(sv->in[1], o, hi);
        TIO<float>::ld4(sv->in[2], o, xi);
      } else {
        TIO<TA>::ld4(sv->in[1], o, xi);
      }
    } else if (VEC && g_in && ahead && ahead->full) {
      IO<TA>::unpack(ahead->a[i], ai);
      IO<XT>::unpack(ahead->x[i], xi);
      if (BWD) IO<float>::ld4(br.h + roff + t, hi);
      if (LOGIN) IO<float>::unpack(ahead->lx[LOGIN ? i : 0], LX + (LOGIN ? 4 * i : 0));
    } else if (VEC && g_in) {
      IO<TA>::ld4(a + t, ai);
      if (BWD) {
        IO<float>::ld4(static_cast<const float*>(xsrc) + roff + t, xi);
        IO<float>::ld4(br.h + roff + t, hi);
        if (LOGIN)
          IO<float>::ld4(static_cast<const float*>(br.x) + roff + t, LX + (LOGIN ? 4 * i : 0));
      } else {
        IO<TA>::ld4(static_cast<const TA*>(xsrc) + roff + t, xi);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t tt = t + e;
        const bool v = tt >= 0 && tt < T;
        ai[e] = v ? IO<TA>::ld1(a + tt) : 0.f;
        if (BWD) {
          xi[e] = v ? IO<float>::ld1(static_cast<const float*>(xsrc) + roff + tt) : 0.f;
          hi[e] = v ? IO<float>::ld1(br.h + roff + tt) : 0.f;
          if (LOGIN)
            LX[LOGIN ? 4 * i + e : 0] =
                v ? IO<float>::ld1(static_cast<const float*>(br.x) + roff + tt) : 0.f;
        } else {
          xi[e] = v ? IO<TA>::ld1(static_cast<const TA*>(xsrc) + roff + tt) : 0.f;
        }
      }
    }
  }

  // this chunk's halos if they came with the look-ahead; then the loads of
  // the next chunk of the row (scan order), before this one is scanned
  const bool had = ahead && ahead->full;
  const float had_ha = had ? ahead->halo_a : 0.f;
  if (ahead) {
    ahead->full = next;
    if (next) {
      const int mn = (S > 0) ? k + 1 : (p.M - 2 - k);
      const int64_t t0n = (int64_t)mn * L - shift;
      const int64_t trn = t0n + (int64_t)V * lane;
      const bool inside_n = t0n >= 0 && t0n + L <= T;  // warp-uniform
#pragma unroll
      for (int i = 0; i < J; ++i) {
        const int64_t t = trn + 4 * i;
        if (VEC && (inside_n || (t >= 0 && t + 4 <= T))) {
          ahead->a[i] = IO<TA>::ldraw(a + t);
          ahead->x[i] = IO<XT>::ldraw(static_cast<const XT*>(xsrc) + roff + t);
          if (LOGIN)
            ahead->lx[LOGIN ? i : 0] = IO<float>::ldraw(static_cast<const float*>(br.x) + roff + t);
        }
      }
      if (BWD) {
        // raw gate halo (log space: log a, -inf outside the row)
        ahead->halo_a = LOGIN ? -CUDART_INF_F : 0.f;
        if (lane == 0) {
          const int64_t pa = (S < 0) ? t0n + L : t0n - 1;
          if (pa >= 0 && pa < T) ahead->halo_a = IO<TA>::ld1(a + pa);
        }
      }
    }
  }

  // backward neighbours across runs: the gate one step past the run's far
  // end in scan order (a_{t+1} for S = -1, a_{t-1} for S = +1) and the
  // state one step past its near end (h_{t-1}, resp. h_{t+1}); the lanes at
  // the chunk's edges take them from memory (the halos)
  float a_nb = 0.f, halo_h = 0.f;
  if (BWD) {
    // log-space backward: the linear adjoint runs on the gates a = exp(log a)
    if (LOGIN) {
#pragma unroll
      for (int e = 0; e < V; ++e) A[e] = __expf(A[e]);
    }
    float halo_a = 0.f;
    if (lane == 0) {
      const int64_t pa = (S < 0) ? t0 + L : t0 - 1;
      const int64_t ph = (S < 0) ? t0 - 1 : t0 + L;
      if (had) {
        halo_a = LOGIN ? __expf(had_ha) : had_ha;
      } else if (pa >= 0 && pa < T) {
        halo_a = LOGIN ? __expf(IO<TA>::ld1(a + pa)) : IO<TA>::ld1(a + pa);
      }
      if (ph >= 0 && ph < T) halo_h = IO<float>::ld1(br.h + roff + ph);  // used after the scan
    }
    halo_a = __shfl_sync(kFull, halo_a, 0);
    const float an = (S < 0) ? __shfl_down_sync(kFull, A[0], 1) : __shfl_up_sync(kFull, A[V - 1], 1);
    a_nb = lane == ((S < 0) ? 31 : 0) ? halo_a : an;
  }
  release();
  // backward: the shifted gate of element e (before sequence cuts), and the
  // neighbouring state that multiplies dx into da
  auto gate_of = [&](int e) -> float {
    if (S < 0) return e + 1 < V ? A[e + 1 < V ? e + 1 : e] : a_nb;
    return e > 0 ? A[e > 0 ? e - 1 : 0] : a_nb;
  };

  // ---- is the run plain: every step valid, no sequence starts or ends in it ----
  int s_run = 0;
  bool plain;
  if (VARLEN) {
    bool all_plain = false;
    if (INSIDE) {
      // warp-uniform: the sequence holding the chunk's first step, searched
      // from lane 0's hint; when it starts before the chunk and the next one
      // starts after its last step, every run of the chunk is plain and in it
      const int s0 = seg_near(win, seg_hint ? __shfl_sync(kFull, *seg_hint, 0) : -1, t0);
      all_plain = (int64_t)win.cu[s0] < t0 && (int64_t)win.cu[s0 + 1] > t0 + L;
      if (all_plain) {
        s_run = s0;
        if (seg_hint) *seg_hint = s0;
      }
    }
    if (all_plain) {
      plain = true;
    } else {
      const int64_t tc = tr < 0 ? 0 : (tr < T ? tr : T - 1);
      s_run = seg_hint ? seg_near(win, *seg_hint, tc) : seg_find(win, tc);
      if (seg_hint) *seg_hint = s_run;
      plain = tr >= 0 && tr + V <= T && (int64_t)win.cu[s_run] != tr &&
              (int64_t)win.cu[s_run + 1] > tr + V;
    }
  } else {
    plain = tr > 0 && tr + V < T;
  }
  // Boundary facts of a valid step tt of the run: does a sequence start or
  // end there, and which row of h0/dh0 belongs to its sequence.
  struct Bound {
    bool start, end;
    int64_t h0row;
  };
  auto bound = [&](int64_t tt) -> Bound {
    Bound b;
    if (VARLEN) {
      const int s = seg_advance(win, s_run, tt);
      b.start = (int64_t)win.cu[s] == tt;
      b.end = (int64_t)win.cu[s + 1] == tt + 1;
      b.h0row = (int64_t)s * p.rows + row;
    } else {
      b.start = tt == 0;
      b.end = tt == T - 1;
      b.h0row = row;
    }
    return b;
  };

  // ---- pass 1: the run's map, composed in scan order ----
  E run = Op::identity();
  if (plain) {
#pragma unroll
    for (int ii = 0; ii < V; ++ii) {
      const int e = (S > 0) ? ii : V - 1 - ii;
      run = Op::compose(run, Op::make(BWD ? gate_of(e) : A[e], X[e]));
    }
  } else {
#pragma unroll
    for (int ii = 0; ii < V; ++ii) {
      const int e = (S > 0) ? ii : V - 1 - ii;
      const int64_t tt = tr + e;
      if (tt < 0 || tt >= T) continue;  // outside the row: the identity
      const Bound bd = bound(tt);
      E v;
      if (!BWD) {
        v = ((S > 0) ? bd.start : bd.end) ? Op::make_first(A[e], X[e], br.h0, bd.h0row)
                                          : Op::make(A[e], X[e]);
      } else {
        // the shifted gate is 0 past the end of the sequence (scan-first step)
        v = Op::make(((S < 0) ? bd.end : bd.start) ? 0.f : gate_of(e), X[e]);
      }
      run = Op::compose(run, v);
    }
  }

  // ---- warp scan of the run maps: exclusive prefix and chunk total ----
  E inc = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const E o = (S > 0) ? Op::shfl_up(inc, off) : Op::shfl_down(inc, off);
    const bool has = (S > 0) ? (lane >= off) : (lane + off < 32);
    if (has) inc = Op::compose(o, inc);
  }
  E ex = (S > 0) ? Op::shfl_up(inc, 1) : Op::shfl_down(inc, 1);
  if (lane == ((S > 0) ? 0 : 31)) ex = Op::identity();
  const E blk = Op::shfl(inc, (S > 0) ? 31 : 0);

  const float c = chunk_carry_in<Op>(p, brn, row, k, stationary, epoch, ticket, blk, carry);

  // ---- pass 2: the recurrence over the run from its carry-in; X[e] becomes
  // the output (h_t forward, the adjoint g_t = dL/dx_t backward) ----
  typename Op::PState st = Op::enter(ex, c);
  if (plain) {
#pragma unroll
    for (int ii = 0; ii < V; ++ii) {
      const int e = (S > 0) ? ii : V - 1 - ii;
      st = Op::step(st, BWD ? gate_of(e) : A[e], X[e]);
      X[e] = Op::out(st);
    }
  } else {
#pragma unroll
    for (int ii = 0; ii < V; ++ii) {
      const int e = (S > 0) ? ii : V - 1 - ii;
      const int64_t tt = tr + e;
      if (tt < 0 || tt >= T) continue;
      const Bound bd = bound(tt);
      if (!BWD) {
        st = ((S > 0) ? bd.start : bd.end) ? Op::first(A[e], X[e], br.h0, bd.h0row)
                                           : Op::step(st, A[e], X[e]);
      } else {
        st = Op::step(st, ((S < 0) ? bd.end : bd.start) ? 0.f : gate_of(e), X[e]);
      }
      X[e] = Op::out(st);
    }
  }

  // ---- stores ----
  const bool staged_out = SMEM && sv->out[0] != nullptr;  // the whole chunk lies inside the row
  if (!BWD) {
    float* h = br.out_h + roff;
#pragma unroll
    for (int i = 0; i < J; ++i) {
      const int64_t t = tr + 4 * i;
      if (staged_out) {
        TIO<float>::st4(sv->out[0], (uint32_t)(t - sv->e0), X + 4 * i);
      } else if (VEC && (INSIDE || (t >= 0 && t + 4 <= T))) {
        IO<float>::st4(h + t, X + 4 * i);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (t + e >= 0 && t + e < T) IO<float>::st1(h + t + e, X[4 * i + e]);
      }
    }
  } else {
    TA* dx = static_cast<TA*>(br.dx) + roff;
    TA* da = static_cast<TA*>(br.da) + roff;
    // the state one step past the run's near end (h_{t-1} for S = -1,
    // h_{t+1} for S = +1), from the neighbour lane or the halo
    halo_h = __shfl_sync(kFull, halo_h, 0);
    const float hx = (S < 0) ? __shfl_up_sync(kFull, H[V - 1], 1) : __shfl_down_sync(kFull, H[0], 1);
    const float h_nb = lane == ((S < 0) ? 0 : 31) ? halo_h : hx;
    auto hn_of = [&](int e) -> float {
      if (S < 0) return e > 0 ? H[e > 0 ? e - 1 : 0] : h_nb;
      return e + 1 < V ? H[e + 1 < V ? e + 1 : e] : h_nb;
    };
#pragma unroll
    for (int i = 0; i < J; ++i) {
      const int64_t t = tr + 4 * i;
      // dx_t = g_t, da_t = g_t h_{t-1}; log-space: d log x_t = g_t x_t and
      // d log a_t = g_t a_t h_{t-1}
      float gx[4], ga[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int idx = 4 * i + e;
        float hn = hn_of(idx);
        const int64_t tt = t + e;
        if (!plain && tt >= 0 && tt < T) {
          // the step that starts the forward recurrence reads h0 and feeds dh0
          // (log space: d log h0 = a_0 g_0 h0)
          const Bound bd = bound(tt);
          if ((S < 0) ? bd.start : bd.end) {
            hn = br.h0 ? (LOGIN ? __expf(br.h0[bd.h0row]) : br.h0[bd.h0row]) : 0.f;
            if (br.dh0) br.dh0[bd.h0row] = A[idx] * X[idx] * (LOGIN ? hn : 1.f);
          }
        }
        ga[e] = X[idx] * hn * (LOGIN ? A[idx] : 1.f);
        gx[e] = LOGIN ? X[idx] * __expf(LX[LOGIN ? idx : 0]) : X[idx];
      }
      if (staged_out) {
        TIO<TA>::st4(sv->out[0], (uint32_t)(t - sv->e0), gx);
        TIO<TA>::st4(sv->out[1], (uint32_t)(t - sv->e0), ga);
      } else if (VEC && (INSIDE || (t >= 0 && t + 4 <= T))) {
        IO<TA>::st4(dx + t, gx);
        IO<TA>::st4(da + t, ga);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (t + e >= 0 && t + e < T) {
            IO<TA>::st1(dx + t + e, gx[e]);
            IO<TA>::st1(da + t + e, ga[e]);
          }
      }
    }
  }
  // this lane's tile writes become visible to the tensor store issued next
  if (staged_out) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <class Op, int MODE, bool VARLEN, bool VEC, int J, typename TA, int S, bool SMEM = false,
          class Release = NoRelease>
__device__ __forceinline__ void chunk(const ScalarParams& p, int brn, int64_t row, int k,
                                      bool stationary, uint32_t epoch, unsigned ticket,
                                      const SegWin& win, float& carry,
                                      const StageView* sv = nullptr, int* seg_hint = nullptr,
                                      const Release& release = Release(),
                                      RunAhead<J, TA, MODE>* ahead = nullptr, bool next = false) {
  if constexpr (!VARLEN && !SMEM && MODE != MODE_LOGBWD && std::is_same<Op, LinOp>::value &&
                sizeof(TA) == 4) {
    chunk_groups<Op, MODE, VEC, J, TA, S>(p, brn, row, k, stationary, epoch, ticket, carry);
    return;
  }
  // Dense forward rows (one scan direction per kernel): a second copy of the
  // chunk code for chunks wholly inside the row, without per-group bounds
  // checks (log-space forward on 8 x 1536 x 4096: 0.115 -> 0.110 ms). Kernels
  // that hold both directions (packed bidirectional rows) or the longer
  // backward body measured slower with the copy (packed forward 1.84 -> 2.13
  // ms, log-space backward 0.200 -> 0.210 ms): instruction-cache pressure.
  if constexpr (VEC && !SMEM && !VARLEN && MODE == MODE_FWD) {
    // the chunk's whole span [t0, t0 + L) inside the row: every group is in it
    const int m = (S > 0) ? k : (p.M - 1 - k);
    const int64_t t0 = (int64_t)m * (128 * J) - (int)((row * p.T) & 3);
    if (t0 >= 0 && t0 + 128 * J <= p.T) {
      chunk_body<Op, MODE, VARLEN, VEC, J, TA, S, SMEM, Release, true>(
          p, brn, row, k, stationary, epoch, ticket, win, carry, sv, seg_hint, release, ahead, next);
      return;
    }
  }
  chunk_body<Op, MODE, VARLEN, VEC, J, TA, S, SMEM, Release, false>(
      p, brn, row, k, stationary, epoch, ticket, win, carry, sv, seg_hint, release, ahead, next);
}

// ---------------------------------------------------------------------------
// tensor copies (TMA) between global and shared memory, and their mbarriers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile(
      "{\n\t.reg .b64 state;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 state, [%0], %1;\n}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// Tile (x, y) of a 2-D tensor map into shared memory; completes on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory tile to tile (x, y) of a 2-D tensor map, in the current bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the newest N bulk groups have finished reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// All bulk groups have completed their global writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar`; false once limit_ns has passed.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t_begin = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t_begin > limit_ns) return false;
  return true;
}

// The stream variant. Warp w of the grid takes rows [w rpw, (w + 1) rpw) of
// the branch-major row list (branch b, row r -> b rows + r) and walks their
// chunks in scan order as one sequence of items, with the carry in registers
// (reset at each row). Lane 0 keeps ns items in flight: each stage of the
// warp's ring receives one item's input tiles by 2-D tensor copies that
// complete on the stage's mbarrier. The warp reads a stage into registers
// and refills it at once with the item ns ahead, so the ring covers only
// the copies' latency and the next rows' first chunks are already arriving
// while a row ends. With out_tiles, a chunk that lies wholly inside its row
// writes its outputs to one of two swizzled output buffers that lane 0 sends
// out with tensor stores (one bulk group per item); other chunks store
// straight from registers.
template <class Op, int MODE, bool VARLEN, int J, typename TA>
__device__ __forceinline__ void stream_rows(const ScalarParams& p, const TmaMaps& maps,
                                            const SegWin& win, unsigned long long* bars,
                                            unsigned char* region) {
  constexpr int L = 128 * J;
  constexpr bool BWD = MODE == MODE_BWD;
  constexpr int EA = (int)sizeof(TA);
  constexpr int E = tma_row_elems(EA);  // flat alignment of a chunk's first step
  constexpr int E1 = tma_row_elems(BWD ? 4 : EA);
  constexpr int EO = tma_row_elems(BWD ? EA : 4);
  constexpr uint32_t kTileA = (uint32_t)tma_tile_bytes(J, EA);
  constexpr uint32_t kTile1 = (uint32_t)tma_tile_bytes(J, BWD ? 4 : EA);
  constexpr uint32_t kStage = (uint32_t)tma_stage_bytes(MODE, J, EA);
  constexpr uint32_t kOut0 = (uint32_t)tma_tile_bytes(J, BWD ? EA : 4);
  constexpr uint32_t kOut = (uint32_t)tma_out_bytes(MODE, J, EA);
  // bytes one item's copies deliver (whole boxes, zero-filled past the end)
  constexpr uint32_t kTx = (uint32_t)L * (BWD ? (uint32_t)EA + 8u : 2u * (uint32_t)EA);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ns = p.ns;
  const bool out_tiles = p.tma_out != 0;
  bars += warp * kMaxStages;
  unsigned char* stages = region + (size_t)warp * tma_warp_bytes(MODE, J, EA, ns, out_tiles);
  unsigned char* outs = stages + (size_t)ns * kStage;

  const int64_t nq = (int64_t)p.nbr * p.rows;
  const int64_t gw = (int64_t)blockIdx.x * p.R + warp;
  const int64_t q0 = gw * p.rpw;
  const int64_t q1 = q0 + p.rpw < nq ? q0 + p.rpw : nq;
  if (q0 >= q1) return;
  const int64_t T = p.T;
  const int M = p.M;

  // a position in the warp's item sequence, advanced one chunk at a time
  struct Cursor {
    int brn, S, k;
    int64_t row, roff, t0;
  };
  auto settle = [&](Cursor& c) {  // derived fields for (brn, row, k)
    c.S = BWD ? -p.br[c.brn].dir : p.br[c.brn].dir;
    c.roff = c.row * T;
    const int m = c.S > 0 ? c.k : M - 1 - c.k;
    c.t0 = (int64_t)m * L - (int64_t)(c.roff & (E - 1));
  };
  auto advance = [&](Cursor& c) {
    if (++c.k == M) {
      c.k = 0;
      if (++c.row == p.rows) {
        c.row = 0;
        ++c.brn;
      }
    }
    settle(c);
  };
  Cursor cur;
  cur.brn = (int)(q0 / p.rows);
  cur.row = q0 % p.rows;
  cur.k = 0;
  settle(cur);
  Cursor nxt = cur;  // next item to issue
  int64_t left = (q1 - q0) * (int64_t)M;  // items not yet issued
  const int64_t n = left;

  auto issue = [&](int s) {  // lane 0: nxt into stage s
    const int64_t f = nxt.roff + nxt.t0;  // flat first element, a multiple of E
    unsigned char* st = stages + (size_t)s * kStage;
    mbar_expect_tx(&bars[s], kTx);
    tma_load_2d(st, &maps.in[nxt.brn][0], 0, (int)(f / E), &bars[s]);
    tma_load_2d(st + kTileA, &maps.in[nxt.brn][1], 0, (int)(f / E1), &bars[s]);
    if (BWD) tma_load_2d(st + kTileA + kTile1, &maps.in[nxt.brn][2], 0, (int)(f / 32), &bars[s]);
  };

  if (lane == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  for (int s = 0; s < ns && left > 0; ++s) {
    if (lane == 0) issue(s);
    advance(nxt);
    --left;
  }
  __syncwarp();

  float carry = 0.f;
  int hint = -1;
  int s = 0;
  unsigned phase = 0;
  for (int64_t i = 0; i < n; ++i) {
    const bool ok = __all_sync(kFull, mbar_wait(&bars[s], phase, p.wait_limit_ns));
    if (!ok) {
      // a copy never landed: record it, give the copies still in flight a
      // bounded chance to finish, and stop this warp
      if (lane == 0) {
        set_status(p.hdr, kStatusTimeout);
        int s2 = s;
        unsigned ph2 = phase;
        for (int64_t j = i + 1; j < n && j < i + ns; ++j) {
          if (++s2 == ns) {
            s2 = 0;
            ph2 ^= 1u;
          }
          mbar_wait(&bars[s2], ph2, p.wait_limit_ns);
        }
      }
      break;
    }
    if (cur.k == 0) {
      carry = BWD ? 0.f : Op::initial_carry();
      hint = -1;
    }
    const bool staged = out_tiles && cur.t0 >= 0 && cur.t0 + L <= T;
    unsigned char* ob = outs + (size_t)(i & 1) * kOut;
    StageView sv;
    const unsigned char* st = stages + (size_t)s * kStage;
    sv.in[0] = st;
    sv.in[1] = st + kTileA;
    sv.in[2] = st + kTileA + kTile1;
    sv.out[0] = staged ? ob : nullptr;
    sv.out[1] = staged ? ob + kOut0 : nullptr;
    sv.e0 = cur.t0;
    sv.c_hi = p.tile_hi - cur.roff;
    if (sv.c_hi > cur.t0 + L) sv.c_hi = cur.t0 + L;
    if (staged) {
      // the tensor store that last read this buffer (two items back) is done
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
    // refill this stage as soon as its tiles are in registers
    const bool refill = left > 0;
    auto release = [&] {
      __syncwarp();
      if (refill && lane == 0) {
        fence_proxy_async_smem();  // the warp's reads of the stage precede the refill
        issue(s);
      }
    };
    if (cur.S > 0)
      chunk<Op, MODE, VARLEN, true, J, TA, 1, true>(p, cur.brn, cur.row, cur.k, true, 0u, 0u, win,
                                                    carry, &sv, &hint, release);
    else
      chunk<Op, MODE, VARLEN, true, J, TA, -1, true>(p, cur.brn, cur.row, cur.k, true, 0u, 0u, win,
                                                     carry, &sv, &hint, release);
    if (refill) {
      advance(nxt);
      --left;
    }
    if (out_tiles) {
      __syncwarp();
      if (lane == 0) {
        if (staged) {
          const int64_t f = cur.roff + cur.t0;
          tma_store_2d(&maps.out[cur.brn][0], 0, (int)(f / EO), ob);
          if (BWD) tma_store_2d(&maps.out[cur.brn][1], 0, (int)(f / E), ob + kOut0);
        }
        bulk_commit();  // one group per item, possibly empty
      }
    }
    advance(cur);
    if (++s == ns) {
      s = 0;
      phase ^= 1u;
    }
  }
  if (out_tiles && lane == 0) bulk_wait_all();
  __syncwarp();
}

// ---------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------

// Packed offsets: staged once per block in shared memory when they fit.
template <bool VARLEN>
__device__ __forceinline__ SegWin stage_offsets(const ScalarParams& p, unsigned char* smem) {
  SegWin win;
  win.cu = p.cu;
  win.n = p.n_seqs;
  if (VARLEN && p.n_seqs + 1 <= kCuSmem) {
    int32_t* s_cu = reinterpret_cast<int32_t*>(smem);
    for (int i = threadIdx.x; i <= p.n_seqs; i += blockDim.x) s_cu[i] = __ldg(p.cu + i);
    __syncthreads();
    win.cu = s_cu;
  }
  return win;
}

template <class Op, int MODE, bool VARLEN, bool VEC, int J, typename TA, int VARIANT>
__device__ __forceinline__ void scalar_scan_body(const ScalarParams& p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const SegWin win = stage_offsets<VARLEN>(p, smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (VARIANT == VAR_LOOKBACK) {
    __shared__ unsigned s_ticket, s_epoch;
    if (threadIdx.x == 0) {
      const unsigned long long te = atomicAdd(&p.hdr->ticket_epoch, 1ull);
      s_ticket = (unsigned)te;
      s_epoch = (unsigned)(te >> 32);
    }
    __syncthreads();
    const unsigned ticket = s_ticket;
    const uint32_t epoch = s_epoch;
    if ((int64_t)ticket < p.ntiles) {
      const int per_k = p.G * p.nbr;
      const int k = (int)(ticket / (unsigned)per_k);
      const int rem = (int)(ticket % (unsigned)per_k);
      const int g = rem / p.nbr;
      const int brn = rem % p.nbr;
      const int64_t row = (int64_t)g * p.R + warp;
      if (VARLEN && ticket == 0) check_segments<MODE>(p);
      float carry = 0.f;
      const int S = (MODE == MODE_FWD) ? p.br[brn].dir : -p.br[brn].dir;
      if (S > 0)
        chunk<Op, MODE, VARLEN, VEC, J, TA, 1>(p, brn, row, k, false, epoch, ticket, win, carry);
      else
        chunk<Op, MODE, VARLEN, VEC, J, TA, -1>(p, brn, row, k, false, epoch, ticket, win, carry);
    } else if (threadIdx.x == 0) {
      set_status(p.hdr, kStatusWorkspace);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned d = atomicAdd(&p.hdr->done, 1u);
      if (d == gridDim.x - 1) finish_lookback_launch(p.hdr, p.recs, p.rec_bytes, epoch);
    }
  } else if (VARIANT == VAR_STATIONARY) {
    // Two branches scan in opposite directions, each through its own copy of
    // the chunk code, and SM pairs (smid 2i, 2i + 1) running both keep twice
    // the code hot. A block takes a row group of the branch matching its SM
    // pair's parity (the other branch once that one is used up: 2 G blocks
    // always find 2 G groups), so an SM pair mostly runs one direction
    // (measured: packed bidirectional backward 3.75 -> 3.31 ms; keying on the
    // SM's own parity instead gained nothing).
    __shared__ int s_g, s_brn;
    if (p.nbr == 2) {
      if (threadIdx.x == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        int b = (int)((smid >> 1) & 1u);
        unsigned tk = atomicAdd(&p.hdr->branch_ticket[b], 1u);
        if (tk >= (unsigned)p.G) {
          b ^= 1;
          tk = atomicAdd(&p.hdr->branch_ticket[b], 1u);
        }
        s_g = (int)tk;
        s_brn = b;
      }
      __syncthreads();
    }
    const int g = p.nbr == 2 ? s_g : blockIdx.x / p.nbr;
    const int brn = p.nbr == 2 ? s_brn : blockIdx.x % p.nbr;
    const int64_t row = (int64_t)g * p.R + warp;
    if (VARLEN && blockIdx.x == 0) check_segments<MODE>(p);
    float carry = (MODE == MODE_FWD) ? Op::initial_carry() : 0.f;
    const int S = (MODE == MODE_FWD) ? p.br[brn].dir : -p.br[brn].dir;
    int hint = -1;
    RunAhead<J, TA, MODE> ahead;
    ahead.full = false;
    RunAhead<J, TA, MODE>* ap = uses_ahead<MODE, VARLEN, TA>() ? &ahead : nullptr;
    for (int k = 0; k < p.M; ++k) {
      const bool next = k + 1 < p.M;
      if (S > 0)
        chunk<Op, MODE, VARLEN, VEC, J, TA, 1>(p, brn, row, k, true, 0u, 0u, win, carry, nullptr,
                                               &hint, NoRelease(), ap, next);
      else
        chunk<Op, MODE, VARLEN, VEC, J, TA, -1>(p, brn, row, k, true, 0u, 0u, win, carry, nullptr,
                                                &hint, NoRelease(), ap, next);
    }
    if (p.nbr == 2) {
      __syncthreads();
      if (threadIdx.x == 0) {
        const unsigned d = atomicAdd(&p.hdr->branch_done, 1u);
        if (d == gridDim.x - 1) {  // every block has taken its ticket and finished
          p.hdr->branch_ticket[0] = 0u;
          p.hdr->branch_ticket[1] = 0u;
          p.hdr->branch_done = 0u;
          __threadfence();
        }
      }
    }
  } else {
    // VAR_SEGMENTED: a row is cut into nseg segments of cps chunks, taken in
    // ticket order (segment index major): a block waits once for the end
    // state of its rows' previous segments (published G * nbr tickets
    // earlier), walks its segment with the carry in registers and publishes
    // its end state.
    __shared__ unsigned s_ticket, s_epoch;
    if (threadIdx.x == 0) {
      const unsigned long long te = atomicAdd(&p.hdr->ticket_epoch, 1ull);
      s_ticket = (unsigned)te;
      s_epoch = (unsigned)(te >> 32);
    }
    __syncthreads();
    const unsigned ticket = s_ticket;
    const uint32_t epoch = s_epoch;
    if ((int64_t)ticket < p.ntiles) {
      const int per_s = p.G * p.nbr;
      const int seg = (int)(ticket / (unsigned)per_s);
      const int rem = (int)(ticket % (unsigned)per_s);
      const int g = rem / p.nbr;
      const int brn = rem % p.nbr;
      if (VARLEN && ticket == 0) check_segments<MODE>(p);
      const int S = (MODE == MODE_FWD) ? p.br[brn].dir : -p.br[brn].dir;
      const int64_t row = (int64_t)g * p.R + warp;
      const bool active = row < p.rows;
      unsigned long long* recs_row = p.recs + ((int64_t)brn * p.rows + row) * (int64_t)p.nseg * 2;
      float carry = (MODE == MODE_FWD) ? Op::initial_carry() : 0.f;
      if (seg > 0 && active) carry = lookback<Op>(p, recs_row, seg, epoch, lane, ticket, brn, row);
      const int k0 = seg * p.cps;
      const int k1 = k0 + p.cps < p.M ? k0 + p.cps : p.M;
      int hint = -1;
      RunAhead<J, TA, MODE> ahead;
      ahead.full = false;
      RunAhead<J, TA, MODE>* ap = uses_ahead<MODE, VARLEN, TA>() ? &ahead : nullptr;
      for (int k = k0; k < k1; ++k) {
        const bool next = k + 1 < k1;
        if (S > 0)
          chunk<Op, MODE, VARLEN, VEC, J, TA, 1>(p, brn, row, k, true, 0u, 0u, win, carry, nullptr,
                                                 &hint, NoRelease(), ap, next);
        else
          chunk<Op, MODE, VARLEN, VEC, J, TA, -1>(p, brn, row, k, true, 0u, 0u, win, carry, nullptr,
                                                  &hint, NoRelease(), ap, next);
      }
      if (active && lane == 0)
        st_relaxed(recs_row + 2 * (int64_t)seg + 1, pack_rec((epoch << 2) | 2u, carry));
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
}

// The register-carry kernels keep ptxas's default register budget for 256-
// thread blocks.
template <class Op, int MODE, bool VARLEN, bool VEC, int J, typename TA, int VARIANT>
__global__ void __launch_bounds__(256) scalar_scan_kernel(const __grid_constant__ ScalarParams p) {
  scalar_scan_body<Op, MODE, VARLEN, VEC, J, TA, VARIANT>(p);
}

// The dense log-space forward waits on memory with a third of the warp slots
// filled at its default 76 registers; held to 64 (four 256-thread blocks per
// SM) it runs 5 % faster on the 8 x 1536 x 4096 rows. (Stating a minimum of
// one block for the other kernels changes their budget too, so they keep the
// form above.)
template <class Op, int MODE, bool VARLEN, bool VEC, int J, typename TA, int VARIANT>
__global__ void __launch_bounds__(256, 4)
    scalar_scan_kernel_r64(const __grid_constant__ ScalarParams p) {
  scalar_scan_body<Op, MODE, VARLEN, VEC, J, TA, VARIANT>(p);
}

template <class Op, int MODE, bool VARLEN>
constexpr bool uses_r64() {
  return std::is_same<Op, LogOp>::value && MODE == MODE_FWD && !VARLEN;
}

// Dense fp32 rows of the linear form, stationary, in chunks of up to 256
// steps: at the default budget (80 registers) 24 row-warps fit an SM, and
// the 12,288 rows of the 8 x 1536 workload take 3.4 waves whose last one
// leaves HBM short of loads in flight. Held to 72 registers (no spills at
// these chunk lengths) 28 fit, 2.9 waves: backward 0.1696 -> 0.1654 ms at
// T = 4096 and 2.562 -> 2.516 ms at T = 65536; forward in chunks of 256
// 1.516 -> 1.464 ms at T = 65536, equal at 4096. (At 64 registers the
// T = 4096 rows lost again; chunks of 512 spill under either cap.)
template <class Op, int MODE, bool VARLEN, bool VEC, int J, typename TA, int VARIANT>
__global__ void __maxnreg__(72) scalar_scan_kernel_r72(const __grid_constant__ ScalarParams p) {
  scalar_scan_body<Op, MODE, VARLEN, VEC, J, TA, VARIANT>(p);
}

// (Not the log-space backward, which runs the linear form's recurrence: its
// vectorised kernel already uses 72 registers at the default budget.)
template <class Op, int MODE, bool VARLEN, int J, typename TA, int VARIANT>
constexpr bool uses_r72() {
  return std::is_same<Op, LinOp>::value && MODE != MODE_LOGBWD && !VARLEN && J <= 2 &&
         std::is_same<TA, float>::value && VARIANT == VAR_STATIONARY;
}

// The stream kernel: persistent warps, occupancy bounded by shared memory.
template <class Op, int MODE, bool VARLEN, int J, typename TA>
__global__ void __launch_bounds__(256, 1)
    scalar_stream_kernel(const __grid_constant__ ScalarParams p, const __grid_constant__ TmaMaps maps) {
  extern __shared__ __align__(16) unsigned char smem[];
  const SegWin win = stage_offsets<VARLEN>(p, smem);
  if (VARLEN && blockIdx.x == 0) check_segments<MODE>(p);
  const size_t cu_bytes = VARLEN ? 4 * (size_t)(p.n_seqs + 1 <= kCuSmem ? p.n_seqs + 1 : 0) : 0;
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem + round_up(cu_bytes, 128));
  const uint32_t base = smem_u32(smem);
  const size_t after = round_up(cu_bytes, 128) + tma_bar_bytes(p.R);
  const size_t pad = (size_t)((1024u - ((base + (uint32_t)after) & 1023u)) & 1023u);
  stream_rows<Op, MODE, VARLEN, J, TA>(p, maps, win, bars, smem + after + pad);
}

// Host-side dispatch over the compile-time choices.
template <class Op, int MODE, typename TA, int VARIANT, bool VARLEN, bool VEC, int J>
cudaError_t launch_one(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  auto kern = [] {  // only the chosen kernel is instantiated
    if constexpr (uses_r64<Op, MODE, VARLEN>())
      return scalar_scan_kernel_r64<Op, MODE, VARLEN, VEC, J, TA, VARIANT>;
    else if constexpr (uses_r72<Op, MODE, VARLEN, J, TA, VARIANT>())
      return scalar_scan_kernel_r72<Op, MODE, VARLEN, VEC, J, TA, VARIANT>;
    else
      return scalar_scan_kernel<Op, MODE, VARLEN, VEC, J, TA, VARIANT>;
  }();
  const size_t smem = pl.smem;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const bool ticketed = VARIANT == VAR_LOOKBACK || VARIANT == VAR_SEGMENTED;
  const int64_t grid = ticketed ? p.ntiles : (int64_t)p.G * p.nbr;
  if (grid <= 0) return cudaSuccess;
  kern<<<(unsigned)grid, 32 * p.R, smem, s>>>(p);
  return cudaGetLastError();
}

// Stream variant: tensor maps for every input and output of each branch, and
// a persistent grid sized by occupancy, rows dealt out evenly to its warps.
template <class Op, int MODE, typename TA, bool VARLEN, int J>
cudaError_t launch_stream(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  constexpr int EA = (int)sizeof(TA);
  auto kern = scalar_stream_kernel<Op, MODE, VARLEN, J, TA>;
  const int64_t n = p.rows * p.T;
  TmaMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  bool ok = true;
  for (int b = 0; b < p.nbr; ++b) {
    const BranchArgs& br = p.br[b];
    ok = ok && encode_tile_map(&maps.in[b][0], br.a, EA, n, J);
    if (MODE == MODE_FWD) {
      ok = ok && encode_tile_map(&maps.in[b][1], br.x, EA, n, J) &&
           encode_tile_map(&maps.out[b][0], br.out_h, 4, n, J);
    } else {
      ok = ok && encode_tile_map(&maps.in[b][1], br.h, 4, n, J) &&
           encode_tile_map(&maps.in[b][2], br.dh, 4, n, J) &&
           encode_tile_map(&maps.out[b][0], br.dx, EA, n, J) &&
           encode_tile_map(&maps.out[b][1], br.da, EA, n, J);
    }
  }
  if (!ok) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * p.R, pl.smem)) !=
      cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  ScalarParams q = p;
  const int64_t nq = (int64_t)p.nbr * p.rows;
  const int64_t warps = (int64_t)per_sm * p.R * sms;
  q.rpw = (int)((nq + warps - 1) / warps);
  const int64_t used = (nq + q.rpw - 1) / q.rpw;
  const int64_t grid = (used + p.R - 1) / p.R;
  constexpr int E = tma_row_elems(EA);
  q.tile_hi = n / E * E;
  if (grid <= 0) return cudaSuccess;
  kern<<<(unsigned)grid, 32 * p.R, pl.smem, s>>>(q, maps);
  return cudaGetLastError();
}

template <class Op, int MODE, typename TA, int VARIANT, bool VARLEN, bool VEC>
cudaError_t launch_pick_j(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  if constexpr (VARIANT == VAR_STREAM) {
    switch (pl.J) {
      case 1: return launch_stream<Op, MODE, TA, VARLEN, 1>(p, pl, s);
      case 2: return launch_stream<Op, MODE, TA, VARLEN, 2>(p, pl, s);
      case 4: return launch_stream<Op, MODE, TA, VARLEN, 4>(p, pl, s);
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (pl.J) {
      case 1: return launch_one<Op, MODE, TA, VARIANT, VARLEN, VEC, 1>(p, pl, s);
      case 2: return launch_one<Op, MODE, TA, VARIANT, VARLEN, VEC, 2>(p, pl, s);
      case 4: return launch_one<Op, MODE, TA, VARIANT, VARLEN, VEC, 4>(p, pl, s);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <class Op, int MODE, typename TA, int VARIANT>
cudaError_t launch_layouts(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  const bool varlen = p.cu != nullptr;
  if constexpr (VARIANT == VAR_STREAM) {  // tensor copies need the vectorised layout
    if constexpr (MODE == MODE_LOGBWD) {
      return cudaErrorInvalidValue;  // planned as stationary
    } else {
      if (!pl.vec) return cudaErrorInvalidValue;
      return varlen ? launch_pick_j<Op, MODE, TA, VARIANT, true, true>(p, pl, s)
                    : launch_pick_j<Op, MODE, TA, VARIANT, false, true>(p, pl, s);
    }
  } else {
    if (varlen)
      return pl.vec ? launch_pick_j<Op, MODE, TA, VARIANT, true, true>(p, pl, s)
                    : launch_pick_j<Op, MODE, TA, VARIANT, true, false>(p, pl, s);
    return pl.vec ? launch_pick_j<Op, MODE, TA, VARIANT, false, true>(p, pl, s)
                  : launch_pick_j<Op, MODE, TA, VARIANT, false, false>(p, pl, s);
  }
}

template <class Op, int MODE, typename TA>
cudaError_t launch_scalar(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  if constexpr (std::is_same<Op, LinOp>::value && (MODE == MODE_FWD || MODE == MODE_BWD))
    if (packed_applies(p, pl, MODE, (int)sizeof(TA)))
      return launch_packed(p, pl, MODE, (int)sizeof(TA), s);
  switch (pl.variant) {
    case VAR_LOOKBACK: return launch_layouts<Op, MODE, TA, VAR_LOOKBACK>(p, pl, s);
    case VAR_STREAM: return launch_layouts<Op, MODE, TA, VAR_STREAM>(p, pl, s);
    case VAR_STATIONARY:
      return p.nseg > 1 ? launch_layouts<Op, MODE, TA, VAR_SEGMENTED>(p, pl, s)
                        : launch_layouts<Op, MODE, TA, VAR_STATIONARY>(p, pl, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace scan
