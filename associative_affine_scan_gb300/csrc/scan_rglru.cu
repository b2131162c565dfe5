// scan_rglru.cu -- RG-LRU gate preparation fused in front of the scalar scan
// ("Our RG-LRU GPU audit": Strengthened fused path -- the recurrent input, two
// gate logits, a_param, an optional segment_pos and initial state; the gate
// activations, log_a, transition, square-root multiplier and write formed in
// registers and never stored, recomputed by the backward, whose square root
// derivative is clipped and whose a_param gradient is reduced from partial
// sums; Exact real chunk algebra -- a reset is a_t = 0 with the canonical
// write). The gate formulas are the method's own; the pages name the tensors
// but do not print them:
//   r_t = sigmoid(gate_a_t), i_t = sigmoid(gate_x_t),
//   log_a_t = 8 r_t log(sigmoid(a_param[c])), a_t = exp(log_a_t),
//   write_t = sqrt(1 - a_t^2) i_t x_t; where segment_pos[b, t] == 0 a_t = 0
//   and write_t = i_t x_t;  h_t = a_t h_{t-1} + write_t, h_{-1} = h0 (or 0).
//
// One warp per row (b, c) walks T in 128-step chunks with the state in a
// register: lane l holds steps 4l .. 4l + 3 of a chunk (one 16-byte vector of
// each input, so every warp access is one coalesced 512-byte run), composes
// their maps (P, Q) and a shuffle scan over the lanes gives each lane its
// carry-in. The forward loads the next chunk's inputs before it computes the
// current one. A block holds the rows of one channel, so the backward sums the
// a_param gradient over b and t in a fixed order, without a workspace. Both
// kernels are held to 64 registers (four 256-thread blocks per SM): on
// 8 x 1536 x 4096 rows the forward ran 0.1505 -> 0.1432 ms, the backward
// (without the forward's look-ahead, which held it at 128 registers) 0.307 ->
// 0.283 ms, a few spilled words included.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "../../include/libscan.h"
#include "scan_internal.h"

namespace scan {
namespace {

constexpr unsigned kRgFull = 0xffffffffu;
constexpr float kRgScale = 8.f;    // log_a = kRgScale r log(sigmoid(a_param))
constexpr float kRgUMin = 1e-6f;   // d sqrt(u) / du is taken at u >= kRgUMin
constexpr int kRgChunk = 128;      // steps per chunk: 4 per lane
constexpr int kRgMaxWarps = 8;     // warps (rows of one channel) per block

struct RgParams {
  const void* x;    // input dtype (fp32 or bf16), as ga, gx and the three gradients below
  const void* ga;   // gate_a logits
  const void* gx;   // gate_x logits
  const float* ap;  // a_param [C]
  const int32_t* seg;  // segment_pos [B, T] or null
  const float* h0;     // [B, C] or null
  float* h;            // forward output / backward input [B, C, T]
  const float* dh;
  void* dx;
  void* dga;
  void* dgx;
  float* dap;  // [C]
  float* dh0;  // [B, C] or null
  int64_t B, C, T;
};

// Per-step gates use the special-function unit (__expf, an approximate
// reciprocal): their few-ulp relative errors scale i, r and 1 - a by
// 1 + O(1e-6), which moves h by about as much, whatever the memory length
// (a long memory sums 1 / (1 - a) steps, each off by (1 - a) 1e-6 at most).
__device__ __forceinline__ float rg_sigmoid(float z) {
  return __fdividef(1.f, 1.f + __expf(-z));
}

// 1 - exp(x) for x <= 0 to a few ulp of itself (x near 0 gives gates near
// 1): for x > -1/8 the series -x (1 + x/2 (1 + x/3 (1 + x/4 (1 + x/5 (1 +
// x/6))))) (the first omitted term is below 1e-9 of the sum), else 1 - e^x.
__device__ __forceinline__ float rg_one_minus_exp(float x) {
  float q = fmaf(x, 1.f / 6.f, 1.f);
  q = fmaf(x * 0.2f, q, 1.f);
  q = fmaf(x * 0.25f, q, 1.f);
  q = fmaf(x * (1.f / 3.f), q, 1.f);
  q = fmaf(x * 0.5f, q, 1.f);
  const float series = -x * q;
  return x > -0.125f ? series : 1.f - __expf(x);
}

// sqrt(u) for u >= 0 from the approximate reciprocal square root
__device__ __forceinline__ float rg_sqrt(float u) { return u > 0.f ? u * rsqrtf(u) : 0.f; }

// log(sigmoid(p)) = -softplus(-p), without overflow for large |p| (once per
// channel: the library's accurate functions)
__device__ __forceinline__ float rg_log_sigmoid(float p) {
  return p < 0.f ? p - log1pf(expf(p)) : -log1pf(expf(-p));
}

// Four consecutive values of a row from step t (zero past T); VEC: t % 4 == 0
// and the row 16-byte aligned, so a whole group is one vector load. FULL: the
// group lies inside the row (no bounds checks).
template <bool VEC, bool FULL>
__device__ __forceinline__ void rg_ld(const float* row, int64_t t, int64_t T, float (&v)[4]) {
  if (VEC && (FULL || t + 4 <= T)) {
    const float4 q = *reinterpret_cast<const float4*>(row + t);
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = FULL || t + j < T ? row[t + j] : 0.f;
  }
}

template <bool VEC, bool FULL>
__device__ __forceinline__ void rg_ld_seg(const int32_t* row, int64_t t, int64_t T, int (&v)[4]) {
  if (!row) {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = 1;
  } else if (VEC && (FULL || t + 4 <= T)) {
    const int4 q = *reinterpret_cast<const int4*>(row + t);
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = FULL || t + j < T ? row[t + j] : 1;
  }
}

template <bool VEC, bool FULL>
__device__ __forceinline__ void rg_st(float* row, int64_t t, int64_t T, const float (&v)[4]) {
  if (VEC && (FULL || t + 4 <= T)) {
    __stcs(reinterpret_cast<float4*>(row + t), make_float4(v[0], v[1], v[2], v[3]));
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (FULL || t + j < T) __stcs(row + t + j, v[j]);
  }
}

// The same for the input dtype TI (fp32 or bf16: 8-byte vectors of 4 bf16,
// rounded to nearest on store).
template <typename TI, bool VEC, bool FULL>
__device__ __forceinline__ void rg_ld_in(const void* base, int64_t off, int64_t t, int64_t T,
                                         float (&v)[4]) {
  const TI* row = static_cast<const TI*>(base) + off;
  if constexpr (std::is_same<TI, float>::value) {
    rg_ld<VEC, FULL>(row, t, T, v);
  } else if (VEC && (FULL || t + 4 <= T)) {
    const uint2 q = *reinterpret_cast<const uint2*>(row + t);
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xffff0000u);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = FULL || t + j < T ? __bfloat162float(row[t + j]) : 0.f;
  }
}

template <typename TI, bool VEC, bool FULL>
__device__ __forceinline__ void rg_st_in(void* base, int64_t off, int64_t t, int64_t T,
                                         const float (&v)[4]) {
  TI* row = static_cast<TI*>(base) + off;
  if constexpr (std::is_same<TI, float>::value) {
    rg_st<VEC, FULL>(row, t, T, v);
  } else if (VEC && (FULL || t + 4 <= T)) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
    __stcs(reinterpret_cast<uint2*>(row + t),
           make_uint2(*reinterpret_cast<const unsigned*>(&lo),
                      *reinterpret_cast<const unsigned*>(&hi)));
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (FULL || t + j < T) row[t + j] = __float2bfloat16_rn(v[j]);
  }
}

// The gate terms of one step: transition a, the write's factors. A reset
// (segment_pos == 0) has a = 0 and multiplier 1.
struct RgStep {
  float a, u, r, i;  // u = 1 - a^2 (multiplier sqrt(u)); u = 1 at a reset
};

// a is formed as 1 - d with d = 1 - a accurate to a few ulp of itself, so
// that a near 1 (long memories) rounds to the nearest fp32 value without a
// bias: the state carries a product of thousands of such gates, and
// exp(log_a) rounded in fp32 came out 0.1 ulp high on average, which
// 23,000-step memories turned into errors of 1e-5 and more. 1 - a^2 = d (2 - d).
__device__ __forceinline__ RgStep rg_gates(float ga, float gx, float ls, bool reset) {
  RgStep s;
  s.i = rg_sigmoid(gx);
  s.r = rg_sigmoid(ga);
  const float d = rg_one_minus_exp(kRgScale * s.r * ls);
  s.a = reset ? 0.f : 1.f - d;
  s.u = reset ? 1.f : d * (2.f - d);
  return s;
}

// One chunk's inputs for one lane (the backward also takes dh and the
// forward's h).
template <bool BWD>
struct RgIn {
  float x[4], ga[4], gx[4];
  int seg[4];
  float dh[BWD ? 4 : 1], h[BWD ? 4 : 1];
};

template <typename TI, bool VEC, bool FULL, bool BWD>
__device__ __forceinline__ void rg_load(const RgParams& p, int64_t base, const int32_t* seg,
                                        int64_t t, RgIn<BWD>& in) {
  rg_ld_in<TI, VEC, FULL>(p.x, base, t, p.T, in.x);
  rg_ld_in<TI, VEC, FULL>(p.ga, base, t, p.T, in.ga);
  rg_ld_in<TI, VEC, FULL>(p.gx, base, t, p.T, in.gx);
  rg_ld_seg<VEC, FULL>(seg, t, p.T, in.seg);
  if constexpr (BWD) {
    rg_ld<VEC, FULL>(p.dh + base, t, p.T, in.dh);
    rg_ld<VEC, FULL>(p.h + base, t, p.T, in.h);
  }
}

// One forward chunk of one row: the lane's four step maps h -> a h + w
// (identity past T), a scan of the lanes' maps, the outputs; carry is the
// state before the chunk, left at the state after it.
template <bool VEC, bool FULL>
__device__ __forceinline__ void rg_fwd_chunk(const RgParams& p, int64_t base, int64_t t,
                                             const RgIn<false>& in, float ls, int lane,
                                             float& carry) {
  const int64_t T = p.T;
  float a[4], w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const RgStep s = rg_gates(in.ga[j], in.gx[j], ls, in.seg[j] == 0);
    const bool valid = FULL || t + j < T;
    a[j] = valid ? s.a : 1.f;
    w[j] = valid ? rg_sqrt(s.u) * s.i * in.x[j] : 0.f;
  }
  float P = a[0], Q = w[0];
#pragma unroll
  for (int j = 1; j < 4; ++j) {
    Q = fmaf(a[j], Q, w[j]);
    P *= a[j];
  }
  // inclusive scan over the lanes (time order): (P, Q) after the lane's run
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float Pu = __shfl_up_sync(kRgFull, P, o), Qu = __shfl_up_sync(kRgFull, Q, o);
    if (lane >= o) {
      Q = fmaf(P, Qu, Q);
      P *= Pu;
    }
  }
  float Pe = __shfl_up_sync(kRgFull, P, 1), Qe = __shfl_up_sync(kRgFull, Q, 1);
  if (lane == 0) {
    Pe = 1.f;
    Qe = 0.f;
  }
  float st = fmaf(Pe, carry, Qe);  // the state before the lane's first step
  float out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    st = fmaf(a[j], st, w[j]);
    out[j] = st;
  }
  rg_st<VEC, FULL>(p.h + base, t, T, out);
  carry = __shfl_sync(kRgFull, st, 31);
}

template <typename TI, bool VEC>
__global__ void __launch_bounds__(32 * kRgMaxWarps, 4) rglru_fwd_kernel(const RgParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t c = blockIdx.x, T = p.T;
  const int64_t nfull = T / kRgChunk;
  const bool tail = T % kRgChunk != 0;
  const float ls = rg_log_sigmoid(p.ap[c]);
  for (int64_t b = warp; b < p.B; b += nw) {
    const int64_t row = b * p.C + c, base = row * T;
    const int32_t* seg = p.seg ? p.seg + b * T : nullptr;
    float carry = p.h0 ? p.h0[row] : 0.f;
    RgIn<false> in, nx;
    if (nfull > 0) rg_load<TI, VEC, true>(p, base, seg, 4 * lane, in);
    else rg_load<TI, VEC, false>(p, base, seg, 4 * lane, in);
    for (int64_t k = 0; k < nfull; ++k) {
      const int64_t t = k * kRgChunk + 4 * lane;
      // the next chunk's loads go out before this one is computed
      if (k + 1 < nfull) rg_load<TI, VEC, true>(p, base, seg, t + kRgChunk, nx);
      else if (tail) rg_load<TI, VEC, false>(p, base, seg, t + kRgChunk, nx);
      rg_fwd_chunk<VEC, true>(p, base, t, in, ls, lane, carry);
      in = nx;
    }
    if (tail) rg_fwd_chunk<VEC, false>(p, base, nfull * kRgChunk + 4 * lane, in, ls, lane, carry);
  }
}

// Backward: the adjoint g_t = dh_t + a_{t+1} g_{t+1} (a_T = 0) from the last
// chunk to the first (lanes still in time order within a chunk), and per step
// dx = g m i, d(gate_x) = g m x i (1 - i), and through a:
//   dL/da = g h_{t-1} + (g i x) (d sqrt(u) / du) (-2 a),  d log_a = a dL/da,
//   d(gate_a) = d log_a * 8 log(sigmoid(a_param)) r (1 - r),
//   d log(sigmoid(a_param)) += d log_a * 8 r;
// a reset step has no gate_a gradient and multiplier 1. h_{t-1} comes from the
// forward output h (h0 before the first step). carry: g at the first step of
// the chunk after this one, left at g at this chunk's first step; a_after: a
// at that step (0 past the end), likewise.
template <typename TI, bool VEC, bool FULL>
__device__ __forceinline__ void rg_bwd_chunk(const RgParams& p, int64_t base, int64_t t0,
                                             RgIn<true>& in, float ls, float init, int lane,
                                             float& carry, float& a_after, float& dls) {
  const int64_t T = p.T, t = t0 + 4 * lane;
  // h_{t-1} before the lane's first step
  float hprev = __shfl_up_sync(kRgFull, in.h[3], 1);
  if (lane == 0) hprev = t0 > 0 ? p.h[base + t0 - 1] : init;
  RgStep s[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    s[j] = rg_gates(in.ga[j], in.gx[j], ls, in.seg[j] == 0);
    if (!FULL && t + j >= T) {
      s[j].a = 0.f;  // past the end: nothing flows back
      in.dh[j] = 0.f;
    }
  }
  // the gate one step later, shifted in from the next lane / chunk
  const float a_nl = __shfl_down_sync(kRgFull, s[0].a, 1);
  const float A[4] = {s[1].a, s[2].a, s[3].a, lane == 31 ? a_after : a_nl};
  // the lane's reverse run: g at its first step = P g_in + Q
  float P = 1.f, Q = 0.f;
#pragma unroll
  for (int j = 3; j >= 0; --j) {
    Q = fmaf(A[j], Q, in.dh[j]);
    P *= A[j];
  }
  // inclusive scan over the lanes in reverse (lanes l .. 31)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float Pd = __shfl_down_sync(kRgFull, P, o), Qd = __shfl_down_sync(kRgFull, Q, o);
    if (lane + o < 32) {
      Q = fmaf(P, Qd, Q);
      P *= Pd;
    }
  }
  float Pe = __shfl_down_sync(kRgFull, P, 1), Qe = __shfl_down_sync(kRgFull, Q, 1);
  if (lane == 31) {
    Pe = 1.f;
    Qe = 0.f;
  }
  float g = fmaf(Pe, carry, Qe);  // g at the step after the lane's run
  float odx[4], oga[4], ogx[4];
#pragma unroll
  for (int j = 3; j >= 0; --j) {
    g = fmaf(A[j], g, in.dh[j]);
    const float hp = j > 0 ? in.h[j > 0 ? j - 1 : 0] : hprev;
    const float xv = in.x[j], ig = s[j].i;
    const bool reset = in.seg[j] == 0;
    const float mult = reset ? 1.f : rg_sqrt(s[j].u);
    odx[j] = g * mult * ig;
    const float d_in = g * mult * xv;
    ogx[j] = d_in * ig * (1.f - ig);
    const float d_mult = g * ig * xv;
    const float dmdu = 0.5f * rsqrtf(fmaxf(s[j].u, kRgUMin));
    const float d_a = fmaf(g, hp, d_mult * dmdu * (-2.f * s[j].a));
    const float dla = (reset || (!FULL && t + j >= T)) ? 0.f : d_a * s[j].a;
    const float r = s[j].r;
    oga[j] = dla * kRgScale * ls * r * (1.f - r);
    dls = fmaf(dla * kRgScale, r, dls);
  }
  rg_st_in<TI, VEC, FULL>(p.dx, base, t, T, odx);
  rg_st_in<TI, VEC, FULL>(p.dga, base, t, T, oga);
  rg_st_in<TI, VEC, FULL>(p.dgx, base, t, T, ogx);
  carry = __shfl_sync(kRgFull, g, 0);  // g at step t0
  a_after = __shfl_sync(kRgFull, s[0].a, 0);
}

template <typename TI, bool VEC>
__global__ void __launch_bounds__(32 * kRgMaxWarps, 4) rglru_bwd_kernel(const RgParams p) {
  __shared__ float s_part[kRgMaxWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t c = blockIdx.x, T = p.T;
  const int64_t nfull = T / kRgChunk;
  const bool tail = T % kRgChunk != 0;
  const float ls = rg_log_sigmoid(p.ap[c]);
  float dls = 0.f;  // this lane's share of dL / d log(sigmoid(a_param[c]))
  for (int64_t b = warp; b < p.B; b += nw) {
    const int64_t row = b * p.C + c, base = row * T;
    const int32_t* seg = p.seg ? p.seg + b * T : nullptr;
    const float init = p.h0 ? p.h0[row] : 0.f;
    float carry = 0.f, a_after = 0.f;
    RgIn<true> in;
    if (tail) {  // the partial last chunk first
      const int64_t t0 = nfull * kRgChunk;
      rg_load<TI, VEC, false>(p, base, seg, t0 + 4 * lane, in);
      rg_bwd_chunk<TI, VEC, false>(p, base, t0, in, ls, init, lane, carry, a_after, dls);
    }
    for (int64_t k = nfull - 1; k >= 0; --k) {
      const int64_t t0 = k * kRgChunk;
      rg_load<TI, VEC, true>(p, base, seg, t0 + 4 * lane, in);
      rg_bwd_chunk<TI, VEC, true>(p, base, t0, in, ls, init, lane, carry, a_after, dls);
    }
    if (p.dh0 && lane == 0) p.dh0[row] = a_after * carry;  // a_0 g_0 (0 when T == 0)
  }
  // the a_param gradient: lanes, then warps, in a fixed order
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) dls += __shfl_xor_sync(kRgFull, dls, o);
  if (lane == 0) s_part[warp] = dls;
  __syncthreads();
  if (threadIdx.x == 0) {
    float sum = 0.f;
    for (int w = 0; w < nw; ++w) sum += s_part[w];
    p.dap[c] = sum * rg_sigmoid(-p.ap[c]);  // d log(sigmoid(p)) / dp = sigmoid(-p)
  }
}

bool aligned(const void* q, size_t n) { return q == nullptr || ((uintptr_t)q % n) == 0; }

template <typename TI>
cudaError_t rg_launch_t(const RgParams& p, bool fwd, bool vec, cudaStream_t s) {
  const int nw = (int)(p.B < kRgMaxWarps ? p.B : kRgMaxWarps);
  const dim3 grid((unsigned)p.C), block(32u * (unsigned)nw);
  if (fwd) {
    if (vec) rglru_fwd_kernel<TI, true><<<grid, block, 0, s>>>(p);
    else rglru_fwd_kernel<TI, false><<<grid, block, 0, s>>>(p);
  } else {
    if (vec) rglru_bwd_kernel<TI, true><<<grid, block, 0, s>>>(p);
    else rglru_bwd_kernel<TI, false><<<grid, block, 0, s>>>(p);
  }
  return cudaGetLastError();
}

// The vector path: rows of T % 4 == 0 elements from base pointers aligned to
// one 4-element vector of their type (16 bytes fp32, 8 bytes bf16).
bool rg_vec(const RgParams& p, scan_dtype dt, bool bwd) {
  const size_t vi = dt == SCAN_BF16 ? 8 : 16;
  bool ok = p.T % 4 == 0 && aligned(p.x, vi) && aligned(p.ga, vi) && aligned(p.gx, vi) &&
            aligned(p.h, 16) && aligned(p.seg, 16);
  if (bwd) ok = ok && aligned(p.dh, 16) && aligned(p.dx, vi) && aligned(p.dga, vi) &&
                aligned(p.dgx, vi);
  return ok;
}

cudaError_t rg_launch(const RgParams& p, scan_dtype dt, bool fwd, cudaStream_t s) {
  const bool vec = rg_vec(p, dt, !fwd);
  return dt == SCAN_BF16 ? rg_launch_t<__nv_bfloat16>(p, fwd, vec, s)
                         : rg_launch_t<float>(p, fwd, vec, s);
}

}  // namespace
}  // namespace scan

using namespace scan;

extern "C" {

scan_status rglru_fwd(const void* x, const void* gate_a, const void* gate_x,
                      const float* a_param, const int32_t* segment_pos, const float* h0, float* h,
                      int64_t B, int64_t C, int64_t T, scan_dtype dt, cudaStream_t stream) {
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  if (B < 0 || C < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (C > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;
  if (B * C * T == 0) return SCAN_OK;
  if (!x || !gate_a || !gate_x || !a_param || !h) return SCAN_ERR_INVALID_ARG;
  RgParams p{};
  p.x = x;
  p.ga = gate_a;
  p.gx = gate_x;
  p.ap = a_param;
  p.seg = segment_pos;
  p.h0 = h0;
  p.h = h;
  p.B = B;
  p.C = C;
  p.T = T;
  return rg_launch(p, dt, true, stream) == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}

scan_status rglru_bwd(const void* x, const void* gate_a, const void* gate_x,
                      const float* a_param, const int32_t* segment_pos, const float* h0,
                      const float* h, const float* dh, void* dx, void* dgate_a, void* dgate_x,
                      float* da_param, float* dh0, int64_t B, int64_t C, int64_t T,
                      scan_dtype dt, cudaStream_t stream) {
  if (dt != SCAN_F32 && dt != SCAN_BF16) return SCAN_ERR_INVALID_ARG;
  if (B < 0 || C < 0 || T < 0) return SCAN_ERR_INVALID_ARG;
  if (C > 0x7fffffffLL) return SCAN_ERR_UNSUPPORTED;
  if (C == 0) return SCAN_OK;
  if (!da_param || !a_param) return SCAN_ERR_INVALID_ARG;
  if (B * T == 0) {  // nothing flows back: the parameter and initial-state gradients are 0
    cudaError_t e = launch_fill_zero(da_param, C, stream);
    if (e == cudaSuccess && dh0) e = launch_fill_zero(dh0, B * C, stream);
    return e == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
  }
  if (!x || !gate_a || !gate_x || !h || !dh || !dx || !dgate_a || !dgate_x)
    return SCAN_ERR_INVALID_ARG;
  RgParams p{};
  p.x = x;
  p.ga = gate_a;
  p.gx = gate_x;
  p.ap = a_param;
  p.seg = segment_pos;
  p.h0 = h0;
  p.h = const_cast<float*>(h);
  p.dh = dh;
  p.dx = dx;
  p.dga = dgate_a;
  p.dgx = dgate_x;
  p.dap = da_param;
  p.dh0 = dh0;
  p.B = B;
  p.C = C;
  p.T = T;
  return rg_launch(p, dt, false, stream) == cudaSuccess ? SCAN_OK : SCAN_ERR_CUDA;
}

}  // extern "C"
