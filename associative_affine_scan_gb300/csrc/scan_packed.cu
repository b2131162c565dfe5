// scan_packed.cu -- the scalar scan over packed rows (cu_seqlens), forward and
// backward, with the carry in registers while one warp walks each row.
//
// The recurrence per sequence ("associative_scan_triton" README, quick start:
// h[t] = g[t] * h[t-1] + x[t] with cu_seqlens, no leakage across sequences;
// the reverse branch runs from each sequence's end) and its backward (how it
// works: a reverse scan of d_tokens on shifted gates, d_gates = shifted_states
// x d_tokens). A sequence start is the constant map (0, a h0 + x) ("Our RG-LRU
// GPU audit", Exact real chunk algebra: a zero gate erases the prefix), so the
// chunk tiling ignores sequence boundaries.
//
// Work decomposition, per warp: one (branch, channel) row, walked chunk by
// chunk (256 steps; each lane owns a run of 8 consecutive steps, loaded as two
// aligned 4-step groups). Per chunk: compose each lane's run map (P, Q), one
// warp-shuffle scan of the 32 run maps, the recurrence over the run from its
// carry-in, vector stores. Forward: each lane copies its runs of the next
// chunks into a per-warp ring in shared memory (cp.async, 3 or 4 chunks deep)
// before it scans the current one; backward: the next chunk's gates and dh
// are loaded into registers before the current one is scanned.
//
// A warp-uniform cursor into cu_seqlens tells whether any sequence boundary
// touches the chunk (a sequence starting in it or right after it) or the
// chunk reaches outside the row: only then do the lanes look up their
// sequences and rewrite the affected element maps (first step of a sequence:
// the constant map; backward: the shifted gate past a sequence's end is 0 and
// the state before its first step is h0). On the benchmark's packed rows
// (64 sequences over 275,479 steps) about 6 % of chunks do; the others run the
// scan with no per-element test. The backward's gate next to the chunk is the
// edge gate of the chunk scanned just before, carried in a register.
#include "scan_scalar.cuh"

namespace scan {
namespace {

constexpr int kPV = 8;         // steps per lane run (two 4-step groups)
constexpr int kPL = 32 * kPV;  // steps per chunk

// First i in [0, n + 1] with cu[i] >= t (n + 1: none), moved from a nearby
// guess i; both walks stay in [0, n + 1] whatever cu holds.
__device__ __forceinline__ int cursor_at(const SegWin& w, int i, int64_t t) {
  while (i > 0 && (int64_t)w.cu[i - 1] >= t) --i;
  while (i <= w.n && (int64_t)w.cu[i] < t) ++i;
  return i;
}

// The 8 values of a lane's run at steps tr .. tr + 7; 0 outside the row.
template <typename TA>
__device__ __forceinline__ void load_run(const TA* base, int64_t tr, int64_t T, bool inside,
                                         float (&v)[kPV]) {
  if (inside) {
    IO<TA>::ld4(base + tr, v);
    IO<TA>::ld4(base + tr + 4, v + 4);
  } else {
#pragma unroll
    for (int e = 0; e < kPV; ++e) {
      const int64_t t = tr + e;
      v[e] = (t >= 0 && t < T) ? IO<TA>::ld1(base + t) : 0.f;
    }
  }
}

template <typename TA>
__device__ __forceinline__ void store_run(TA* base, int64_t tr, int64_t T, bool inside,
                                          const float (&v)[kPV]) {
  if (inside) {
    IO<TA>::st4(base + tr, v);
    IO<TA>::st4(base + tr + 4, v + 4);
  } else {
#pragma unroll
    for (int e = 0; e < kPV; ++e) {
      const int64_t t = tr + e;
      if (t >= 0 && t < T) IO<TA>::st1(base + t, v[e]);
    }
  }
}

// Scan of the lanes' run maps in scan order S (+1: lane 0 first, -1: lane 31
// first): the exclusive prefix of this lane and the chunk's total.
template <int S>
__device__ __forceinline__ void warp_scan(LinOp::E run, int lane, LinOp::E& ex, LinOp::E& tot) {
  LinOp::E inc = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const LinOp::E o = (S > 0) ? LinOp::shfl_up(inc, off) : LinOp::shfl_down(inc, off);
    if ((S > 0) ? (lane >= off) : (lane + off < 32)) inc = LinOp::compose(o, inc);
  }
  ex = (S > 0) ? LinOp::shfl_up(inc, 1) : LinOp::shfl_down(inc, 1);
  if (lane == ((S > 0) ? 0 : 31)) ex = LinOp::identity();
  tot = LinOp::shfl(inc, (S > 0) ? 31 : 0);
}

// Asynchronous 8- or 16-byte copies from global to shared memory, one commit
// group per chunk.
template <int N>
__device__ __forceinline__ void cp_async(void* dst, const void* src) {
  if constexpr (N == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "n"(N)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A warp's ring of D chunk slots in shared memory: each lane copies its run's
// two 4-step groups of both tensors into its own entries (U: gates, W: x or
// dh), D - 1 chunks ahead of the one it scans, and reads them back when that
// chunk comes (no registers held for loads in flight). Chunks that reach out
// of the row are loaded directly instead (their slot stays unused).
template <typename TU, typename TW>
struct Ring {
  static constexpr int EU = 4 * (int)sizeof(TU), EW = 4 * (int)sizeof(TW);  // bytes per group
  static constexpr int SLOT = 32 * 2 * (EU + EW);
  static constexpr int D = SLOT <= 1536 ? 4 : 3;  // chunks in the ring
  static constexpr int BYTES = D * SLOT;          // per warp
  unsigned char* base;
  __device__ __forceinline__ unsigned char* u(int k, int i, int lane) const {
    return base + (k % D) * SLOT + (i * 32 + lane) * EU;
  }
  __device__ __forceinline__ unsigned char* w(int k, int i, int lane) const {
    return base + (k % D) * SLOT + 64 * EU + (i * 32 + lane) * EW;
  }
  // copies of chunk k (when it lies inside the row; tr its lane's run start)
  __device__ __forceinline__ void issue(int k, bool inside, int64_t tr, const TU* u0,
                                        const TW* w0, int lane) const {
    if (inside) {
      cp_async<EU>(u(k, 0, lane), u0 + tr);
      cp_async<EU>(u(k, 1, lane), u0 + tr + 4);
      cp_async<EW>(w(k, 0, lane), w0 + tr);
      cp_async<EW>(w(k, 1, lane), w0 + tr + 4);
    }
    cp_async_commit();
  }
  __device__ __forceinline__ void read(int k, int lane, float (&U)[8], float (&W)[8]) const {
    IO<TU>::unpack(*reinterpret_cast<const typename IO<TU>::Raw*>(u(k, 0, lane)), U);
    IO<TU>::unpack(*reinterpret_cast<const typename IO<TU>::Raw*>(u(k, 1, lane)), U + 4);
    IO<TW>::unpack(*reinterpret_cast<const typename IO<TW>::Raw*>(w(k, 0, lane)), W);
    IO<TW>::unpack(*reinterpret_cast<const typename IO<TW>::Raw*>(w(k, 1, lane)), W + 4);
  }
};

template <typename TA>
using PackedRing = Ring<TA, TA>;  // forward: gates and x

template <typename TA, int MODE>
constexpr size_t ring_bytes() {
  return MODE == MODE_FWD ? (size_t)PackedRing<TA>::BYTES : 0;
}

// ---------------------------------------------------------------------------
// forward: h_t = a_t h_{t-S} + x_t, scanned in direction S
// ---------------------------------------------------------------------------

template <typename TA, int S>
__device__ void packed_fwd_row(const ScalarParams& p, const BranchArgs& br, int64_t row,
                               const SegWin& win, int lane, unsigned char* ring_base) {
  const int64_t T = p.T, roff = row * T;
  const int shift = (int)(roff & 3);  // 4-step groups on 4-element boundaries of memory
  const TA* a = static_cast<const TA*>(br.a) + roff;
  const TA* x = static_cast<const TA*>(br.x) + roff;
  float* h = br.out_h + roff;
  const int M = p.M;
  using R = PackedRing<TA>;
  const R ring{ring_base};
  auto t0_of = [&](int k) { return (int64_t)((S > 0) ? k : (M - 1 - k)) * kPL - shift; };
  auto inside_at = [&](int64_t t) { return t >= 0 && t + kPL <= T; };
  auto issue = [&](int k) {
    const int64_t t0k = k < M ? t0_of(k) : -1;
    ring.issue(k, k < M && inside_at(t0k), t0k + kPV * lane, a, x, lane);
  };
  for (int k = 0; k < R::D - 1; ++k) issue(k);
  float carry = 0.f;
  int cur = (S > 0) ? 0 : win.n;
  for (int k = 0; k < M; ++k) {
    const int64_t t0 = t0_of(k);
    const bool ins = inside_at(t0);
    const int64_t tr = t0 + kPV * lane;
    issue(k + R::D - 1);  // into the slot of chunk k - 1, already read
    cp_async_wait<R::D - 1>();
    float A[kPV], X[kPV];
    if (ins) {
      ring.read(k, lane, A, X);
    } else {
      load_run(a, tr, T, false, A);
      load_run(x, tr, T, false, X);
    }
    // boundaries: a sequence starting in [t0, t0 + L] or a chunk reaching out of the row
    cur = cursor_at(win, cur, t0);
    if (!ins || (cur <= win.n && (int64_t)win.cu[cur] <= t0 + kPL)) {
      const int64_t tc = tr < 0 ? 0 : (tr < T ? tr : T - 1);
      int s = seg_find(win, tc);
#pragma unroll
      for (int e = 0; e < kPV; ++e) {
        const int64_t t = tr + e;
        if (t < 0 || t >= T) {  // outside the row: the identity, not written
          A[e] = 1.f, X[e] = 0.f;
          continue;
        }
        s = seg_advance(win, s, t);
        const bool first = (S > 0) ? (int64_t)win.cu[s] == t : (int64_t)win.cu[s + 1] == t + 1;
        if (first) {
          X[e] = fmaf(A[e], br.h0 ? br.h0[(int64_t)s * p.rows + row] : 0.f, X[e]);
          A[e] = 0.f;
        }
      }
    }
    // the run's map in scan order, the warp scan, the recurrence from the carry-in
    LinOp::E run = LinOp::identity();
#pragma unroll
    for (int ii = 0; ii < kPV; ++ii) {
      const int e = (S > 0) ? ii : kPV - 1 - ii;
      run = LinOp::compose(run, LinOp::make(A[e], X[e]));
    }
    LinOp::E ex, tot;
    warp_scan<S>(run, lane, ex, tot);
    const float c = carry;
    carry = fmaf(tot.p, c, tot.q);
    float st = fmaf(ex.p, c, ex.q);
#pragma unroll
    for (int ii = 0; ii < kPV; ++ii) {
      const int e = (S > 0) ? ii : kPV - 1 - ii;
      st = fmaf(A[e], st, X[e]);
      X[e] = st;
    }
    store_run(h, tr, T, ins, X);
  }
}

// ---------------------------------------------------------------------------
// backward of the recurrence running in direction D (scan direction S = -D):
// g_t = dh_t + a'_{t+D} g_{t+D}, dx_t = g_t, da_t = g_t h_{t-D}, dh0 = a g at
// each sequence's first step; a'_{t+D} = 0 past a sequence's last step
// ---------------------------------------------------------------------------

template <typename TA, int D>
__device__ void packed_bwd_row(const ScalarParams& p, const BranchArgs& br, int64_t row,
                               const SegWin& win, int lane) {
  constexpr int S = -D;
  // (the next chunk's gates and dh are held in registers: a shared-memory
  // ring here, 3 or 4 chunks deep with or without the states h, measured
  // slower, 2.69 -> 2.85 / 3.67 ms on the 64-sequence rows)
  const int64_t T = p.T, roff = row * T;
  const int shift = (int)(roff & 3);
  const TA* a = static_cast<const TA*>(br.a) + roff;
  const float* hs = br.h + roff;
  const float* dh = br.dh + roff;
  TA* dx = static_cast<TA*>(br.dx) + roff;
  TA* da = static_cast<TA*>(br.da) + roff;
  const int M = p.M;
  auto t0_of = [&](int k) { return (int64_t)((S > 0) ? k : (M - 1 - k)) * kPL - shift; };
  auto inside_at = [&](int64_t t) { return t >= 0 && t + kPL <= T; };
  typename IO<TA>::Raw ra[2];
  float4 rd[2];
  int64_t t0 = t0_of(0);
  bool ins = inside_at(t0);
  if (ins) {
    const int64_t tr = t0 + kPV * lane;
    ra[0] = IO<TA>::ldraw(a + tr), ra[1] = IO<TA>::ldraw(a + tr + 4);
    rd[0] = IO<float>::ldraw(dh + tr), rd[1] = IO<float>::ldraw(dh + tr + 4);
  }
  float carry = 0.f;
  float gate_carry = 0.f;  // the gate next to the chunk in scan order (0 outside the row)
  int cur = (S > 0) ? 0 : win.n;
  for (int k = 0; k < M; ++k) {
    const int64_t tr = t0 + kPV * lane;
    float A[kPV], G[kPV], H[kPV];
    if (ins) {
      IO<TA>::unpack(ra[0], A), IO<TA>::unpack(ra[1], A + 4);
      IO<float>::unpack(rd[0], G), IO<float>::unpack(rd[1], G + 4);
    } else {
      load_run(a, tr, T, false, A);
      load_run(dh, tr, T, false, G);
    }
    load_run(hs, tr, T, ins, H);  // used after the scan
    // the state next to the chunk on the side of the recurrence's past
    float hh = 0.f;
    if (lane == 0) {
      const int64_t ph = (D > 0) ? t0 - 1 : t0 + kPL;
      if (ph >= 0 && ph < T) hh = IO<float>::ld1(hs + ph);
    }
    int64_t t0n = 0;
    bool insn = false;
    if (k + 1 < M) {
      t0n = t0_of(k + 1);
      insn = inside_at(t0n);
      if (insn) {
        const int64_t trn = t0n + kPV * lane;
        ra[0] = IO<TA>::ldraw(a + trn), ra[1] = IO<TA>::ldraw(a + trn + 4);
        rd[0] = IO<float>::ldraw(dh + trn), rd[1] = IO<float>::ldraw(dh + trn + 4);
      }
    }
    // shifted gates a_{t+D}: inside the run, from the neighbouring lane, or at
    // the chunk's edge the gate carried from the chunk scanned before
    float gate[kPV];
    {
      const float nb = (D > 0) ? __shfl_down_sync(kFull, A[0], 1) : __shfl_up_sync(kFull, A[kPV - 1], 1);
      const bool edge = lane == ((D > 0) ? 31 : 0);
#pragma unroll
      for (int e = 0; e < kPV; ++e) {
        if (D > 0) gate[e] = e + 1 < kPV ? A[e + 1 < kPV ? e + 1 : e] : (edge ? gate_carry : nb);
        else gate[e] = e > 0 ? A[e > 0 ? e - 1 : 0] : (edge ? gate_carry : nb);
      }
      // the next chunk (below for D > 0, above for D < 0) borders this one's
      // first (resp. last) step
      gate_carry = (D > 0) ? __shfl_sync(kFull, A[0], 0) : __shfl_sync(kFull, A[kPV - 1], 31);
    }
    // sequence boundaries: the gate past a sequence's last step (in the
    // recurrence's order) is 0; its first step's previous state is h0 (set
    // after the scan, with dh0)
    unsigned first_mask = 0u;
    int s_first = 0;
    cur = cursor_at(win, cur, t0);
    const bool special = !ins || (cur <= win.n && (int64_t)win.cu[cur] <= t0 + kPL);
    if (special) {
      const int64_t tc = tr < 0 ? 0 : (tr < T ? tr : T - 1);
      int s = seg_find(win, tc);
      s_first = s;
#pragma unroll
      for (int e = 0; e < kPV; ++e) {
        const int64_t t = tr + e;
        if (t < 0 || t >= T) {  // outside the row: the identity, not written
          gate[e] = 1.f, G[e] = 0.f;
          continue;
        }
        s = seg_advance(win, s, t);
        const bool at_lo = (int64_t)win.cu[s] == t, at_hi = (int64_t)win.cu[s + 1] == t + 1;
        if ((D > 0) ? at_hi : at_lo) gate[e] = 0.f;
        if ((D > 0) ? at_lo : at_hi) first_mask |= 1u << e;
      }
    }
    LinOp::E run = LinOp::identity();
#pragma unroll
    for (int ii = 0; ii < kPV; ++ii) {
      const int e = (S > 0) ? ii : kPV - 1 - ii;
      run = LinOp::compose(run, LinOp::make(gate[e], G[e]));
    }
    LinOp::E ex, tot;
    warp_scan<S>(run, lane, ex, tot);
    const float c = carry;
    carry = fmaf(tot.p, c, tot.q);
    float st = fmaf(ex.p, c, ex.q);
#pragma unroll
    for (int ii = 0; ii < kPV; ++ii) {
      const int e = (S > 0) ? ii : kPV - 1 - ii;
      st = fmaf(gate[e], st, G[e]);
      G[e] = st;
    }
    // da_t = g_t h_{t-D}: inside the run, from the neighbouring lane, or the halo
    float DA[kPV];
    {
      const float nb = (D > 0) ? __shfl_up_sync(kFull, H[kPV - 1], 1) : __shfl_down_sync(kFull, H[0], 1);
      const float halo = __shfl_sync(kFull, hh, 0);
      const bool edge = lane == ((D > 0) ? 0 : 31);
#pragma unroll
      for (int e = 0; e < kPV; ++e) {
        float hp;
        if (D > 0) hp = e > 0 ? H[e > 0 ? e - 1 : 0] : (edge ? halo : nb);
        else hp = e + 1 < kPV ? H[e + 1 < kPV ? e + 1 : e] : (edge ? halo : nb);
        DA[e] = G[e] * hp;
      }
    }
    // a sequence's first step: the previous state is h0, and dh0 = a g there
    if (first_mask) {
      int s = s_first;
#pragma unroll
      for (int e = 0; e < kPV; ++e) {
        const int64_t t = tr + e;
        if (!(first_mask & (1u << e))) continue;
        s = seg_advance(win, s, t);
        const int64_t i0 = (int64_t)s * p.rows + row;
        DA[e] = G[e] * (br.h0 ? br.h0[i0] : 0.f);
        if (br.dh0) br.dh0[i0] = IO<TA>::ld1(a + t) * G[e];
      }
    }
    store_run(dx, tr, T, ins, G);
    store_run(da, tr, T, ins, DA);
    t0 = t0n;
    ins = insn;
  }
}

// One warp per (branch, row). Two-branch launches take their row group from a
// per-branch ticket chosen by the parity of the block's SM pair, as the
// register-carry kernels do, so an SM pair mostly runs one scan direction.
// Bytes of the packed offsets staged at the start of dynamic shared memory,
// rounded up to 16 (the rings follow).
__host__ __device__ __forceinline__ size_t cu_smem_bytes(const ScalarParams& p) {
  return round_up(p.cu && p.n_seqs + 1 <= kCuSmem ? 4 * (size_t)(p.n_seqs + 1) : 0, 16);
}

// At most 72 registers: 28 row-warps per SM, so the 4096 row-warps of the
// packed bidirectional workload (2 x 2048 rows) are all resident in one wave;
// a second wave would double the walk.
template <typename TA, int MODE>
__global__ void __maxnreg__(72) packed_kernel(const __grid_constant__ ScalarParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  // dense rows are packed rows with one sequence each: offsets {0, T}, h0 and
  // dh0 indexed by row
  __shared__ int32_t s_dense_cu[2];
  SegWin win;
  if (p.cu) {
    win = stage_offsets<true>(p, smem);
  } else {
    if (threadIdx.x == 0) {
      s_dense_cu[0] = 0;
      s_dense_cu[1] = (int32_t)p.T;
    }
    __syncthreads();
    win.cu = s_dense_cu;
    win.n = 1;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  const int g = p.nbr == 2 ? s_g : (int)blockIdx.x;
  const int brn = p.nbr == 2 ? s_brn : 0;
  if (p.cu && blockIdx.x == 0) check_segments<MODE>(p);
  const int64_t row = (int64_t)g * p.R + warp;
  if (row < p.rows) {
    const BranchArgs& br = p.br[brn];
    // this warp's ring follows the staged offsets in dynamic shared memory
    unsigned char* ring = smem + cu_smem_bytes(p) + (size_t)warp * ring_bytes<TA, MODE>();
    if (MODE == MODE_FWD) {
      if (br.dir > 0) packed_fwd_row<TA, 1>(p, br, row, win, lane, ring);
      else packed_fwd_row<TA, -1>(p, br, row, win, lane, ring);
    } else {
      if (br.dir > 0) packed_bwd_row<TA, 1>(p, br, row, win, lane);
      else packed_bwd_row<TA, -1>(p, br, row, win, lane);
    }
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
}

template <typename TA, int MODE>
cudaError_t launch_packed_t(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s) {
  auto kern = packed_kernel<TA, MODE>;
  const int64_t grid = (int64_t)p.G * p.nbr;
  if (grid <= 0) return cudaSuccess;
  const size_t smem = cu_smem_bytes(p) + (size_t)p.R * ring_bytes<TA, MODE>();
  // above the default 48 KB per block (static shared memory included) the
  // kernel must opt in
  if (smem + 1024 > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)grid, 32 * p.R, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Packed rows, and the backward of dense bf16 rows (8 x 1536 x 4096: 0.1373 ->
// 0.1274 ms). Dense fp32 rows keep the interleaved kernels (the forward here
// measured 0.149 against 0.102 ms), the dense bf16 forward its 512-step lane
// runs.
bool packed_applies(const ScalarParams& p, const ScalarPlan& pl, int mode, int elt) {
  const bool rows = p.cu != nullptr || (elt == 2 && mode == MODE_BWD && p.T <= 0x7fffffffLL);
  return rows && pl.vec && pl.variant == VAR_STATIONARY && p.nseg == 1 && pl.J == 2 && p.R <= 8;
}

cudaError_t launch_packed(const ScalarParams& p, const ScalarPlan& pl, int mode, int elt,
                          cudaStream_t s) {
  if (elt == 4)
    return mode == MODE_FWD ? launch_packed_t<float, MODE_FWD>(p, pl, s)
                            : launch_packed_t<float, MODE_BWD>(p, pl, s);
  return mode == MODE_FWD ? launch_packed_t<__nv_bfloat16, MODE_FWD>(p, pl, s)
                          : launch_packed_t<__nv_bfloat16, MODE_BWD>(p, pl, s);
}

}  // namespace scan
