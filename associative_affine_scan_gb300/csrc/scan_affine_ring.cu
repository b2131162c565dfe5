// scan_affine_ring.cu -- the 4 x 4 block scan for lane-rich shapes: each
// (b, n) lane walks all of T with its state in registers, fed by a ring of
// tensor copies.
//
// H_t = A_t H_{t-1} + B_t with 4 x 4 blocks ("Triton scan kernels", One
// associative-scan family: A_t is k x k, B_t and H_t are k x v; Kernel design:
// one (b, n) lane per state block walks T), and its backward ("Autograd
// integration and the reversed-scan backward"): G_t = dH_t + A_{t+1}^T
// G_{t+1}, dB_t = G_t, dA_t = G_t H_{t-1}^T, dh0 = A_0^T G_0.
//
// One warp (the whole block) owns 8 consecutive lanes n0 .. n0 + 7 of one
// batch row b; thread 4 l + j owns column j of lane n0 + l's state (H_t[:, j]
// forward, G_t[:, j] backward). A column evolves on its own given A_t:
// H_t[:, j] = A_t H_{t-1}[:, j] + B_t[:, j], so the forward needs no exchange
// between threads; the backward's dA_t = G_t H_{t-1}^T sums over the four
// columns, a reduce-scatter by shuffles that leaves row j of dA_t in thread j.
//
// Memory: a 4-D tensor map views each [B, T, N, 4, 4] tensor as {16 floats,
// N lanes, T steps, B} with the 64-byte swizzle. A stage holds LC steps of the
// warp's 8 lanes of each input (LC x 512 bytes per tensor); lane 0 keeps NS
// stages of tensor copies in flight on per-stage mbarriers, refilling a stage
// as soon as the warp has read it. With the swizzle, the 16-byte piece q of
// lane l's 64-byte block sits at piece q ^ ((l >> 1) & 3), so the eight lanes'
// pieces of one row (or one column's elements) fall in eight different bank
// groups: every shared-memory access of a step is conflict-free. Outputs are
// written to swizzled tiles of the same shape and leave by tensor stores, two
// tiles in flight per output. Every global access is a whole-tile tensor copy
// (coalesced; lanes past N and steps past T are zero-filled on load and
// clipped on store).
//
// Bounded waits: an mbarrier wait that passes wait_limit_ns records
// SCAN_ERR_TIMEOUT in the workspace header, waits (bounded) for the copies the
// warp still has in flight and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "scan_scalar.cuh"

namespace scan {
namespace {

constexpr int kRingLanes = 8;      // lanes per warp (4 column threads each)
constexpr int kRingLC = 16;        // steps per stage
constexpr int kRingStagesFwd = 5;  // input stages in flight, forward (A, B)
constexpr int kRingStagesBwd = 3;  // backward (A, H, dH)
constexpr unsigned kTile = kRingLC * kRingLanes * 64;  // bytes per tensor per stage

struct RingParams {
  CUtensorMap in[3];   // forward: A, B; backward: A, H, dH
  CUtensorMap out[2];  // forward: H; backward: dA, dB
  const float* A;      // backward: A_0 for dh0
  const float* h0;     // nullable initial state [B, N, 4, 4]
  float* dh0;          // backward, nullable
  int64_t B, T, N;
  int gpb;             // lane groups per batch row: ceil(N / 8)
  int nchunks;         // ceil(T / LC)
  WsHeader* hdr;
  unsigned long long wait_limit_ns;
  int test_stall;
};

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, int x, int y, int z, int w,
                                             const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::
          "l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(src))
      : "memory");
}

__device__ __forceinline__ float comp(const float4& v, int r) {
  return r == 0 ? v.x : (r == 1 ? v.y : (r == 2 ? v.z : v.w));
}

// Drains what the warp has in flight after a failed wait: the loads of
// chunks [from, to) (bounded waits) and every tensor store.
template <int NS>
__device__ void drain(unsigned long long* bars, int from, int to, unsigned long long limit) {
  for (int u = from; u < to; ++u) (void)mbar_wait(&bars[u % NS], (unsigned)((u / NS) & 1), limit);
  bulk_wait_all();
}

__device__ void record_timeout(const RingParams& p, int chunk) {
  set_status(p.hdr, kStatusTimeout);
  p.hdr->info[0] = blockIdx.x;
  p.hdr->info[1] = 0u;
  p.hdr->info[2] = 0u;
  p.hdr->info[3] = (unsigned)chunk;
}

// The dynamic shared memory, rounded up to the 1024-byte boundary the swizzle
// pattern repeats on. The offset is added to the __shared__ array itself, so
// every pointer derived from it stays a shared-memory pointer.
__device__ __forceinline__ unsigned char* ring_base(unsigned char* smem) {
  const uint32_t pad = (1024u - (smem_u32(smem) & 1023u)) & 1023u;
  return smem + pad;
}

template <typename T>
__device__ __forceinline__ T lds(const unsigned char* base, int off) {
  return *reinterpret_cast<const T*>(base + off);
}
template <typename T>
__device__ __forceinline__ void sts(unsigned char* base, int off, T v) {
  *reinterpret_cast<T*>(base + off) = v;
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

// One step i of a stage: column j of H_t = A_t H_{t-1} + B_t. offA[q]: piece
// q (row q of A) of this lane's block; offC[r]: element j of row r.
__device__ __forceinline__ void fwd_step(const unsigned char* As, const unsigned char* Bs,
                                         unsigned char* Os, int i, const int (&offA)[4],
                                         const int (&offC)[4], float (&h)[4]) {
  const int base = i * 512;
  float4 a[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) a[q] = lds<float4>(As, base + offA[q]);
  float hn[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float bc = lds<float>(Bs, base + offC[r]);
    hn[r] = fmaf(a[r].w, h[3], fmaf(a[r].z, h[2], fmaf(a[r].y, h[1], fmaf(a[r].x, h[0], bc))));
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    h[r] = hn[r];
    sts<float>(Os, base + offC[r], hn[r]);
  }
}

__global__ void __launch_bounds__(32) affine44_ring_fwd(const __grid_constant__ RingParams p) {
  constexpr int NS = kRingStagesFwd;
  extern __shared__ unsigned char ring_smem[];
  __shared__ unsigned long long bars[NS + 1];  // + one that nothing completes (test stall)
  const int lane = threadIdx.x, l = lane >> 2, j = lane & 3;
  const int b = blockIdx.x / p.gpb;
  const int n0 = (blockIdx.x % p.gpb) * kRingLanes;
  const int64_t n = n0 + l;
  unsigned char* stage0 = ring_base(ring_smem);
  unsigned char* out0 = stage0 + (size_t)NS * 2 * kTile;
  const int nch = p.nchunks;
  auto issue = [&](int c) {
    const int s = c % NS;
    unsigned char* st = stage0 + (size_t)s * 2 * kTile;
    mbar_expect_tx(&bars[s], 2 * kTile);
    tma_load_4d(st, &p.in[0], 0, n0, c * kRingLC, b, &bars[s]);
    tma_load_4d(st + kTile, &p.in[1], 0, n0, c * kRingLC, b, &bars[s]);
  };
  if (lane == 0) {
    for (int s = 0; s <= NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    for (int c = 0; c < NS && c < nch; ++c) issue(c);
  }
  __syncwarp();

  const int sl = (l >> 1) & 3;
  int offA[4], offC[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    offA[q] = l * 64 + ((q ^ sl) << 4);
    offC[q] = offA[q] + 4 * j;
  }
  // column j of the state: H[i][j], i = 0..3
  float h[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.h0 && n < p.N) {
    const float* h0 = p.h0 + ((int64_t)b * p.N + n) * 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = h0[i * 4 + j];
  }

  for (int c = 0; c < nch; ++c) {
    const int s = c % NS;
    unsigned long long* bar = (p.test_stall && blockIdx.x == 0 && c == 1) ? &bars[NS] : &bars[s];
    if (!mbar_wait(bar, (unsigned)((c / NS) & 1), p.wait_limit_ns)) {
      if (lane == 0) {
        record_timeout(p, c);
        drain<NS>(bars, c, (c + NS < nch ? c + NS : nch), p.wait_limit_ns);
      }
      return;
    }
    // the tensor store that used this output buffer two chunks ago has read it
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    const unsigned char* As = stage0 + (size_t)s * 2 * kTile;
    const unsigned char* Bs = As + kTile;
    unsigned char* Os = out0 + (size_t)(c & 1) * kTile;
    const int64_t t0 = (int64_t)c * kRingLC;
    const int steps = p.T - t0 < kRingLC ? (int)(p.T - t0) : kRingLC;
    if (steps == kRingLC) {
#pragma unroll
      for (int i = 0; i < kRingLC; ++i) fwd_step(As, Bs, Os, i, offA, offC, h);
    } else {
      for (int i = 0; i < steps; ++i) fwd_step(As, Bs, Os, i, offA, offC, h);
    }
    // the warp's reads of stage s and writes of the output tile are done
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_4d(&p.out[0], 0, n0, (int)t0, b, Os);
      bulk_commit();
      if (c + NS < nch) issue(c + NS);
    }
  }
  if (lane == 0) bulk_wait_all();
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------

// One step i of a stage (t = t0 + i): column j of G_t = dH_t + A_{t+1}^T
// G_{t+1} (g: column j of G_{t+1} on entry, of G_t on return), column j of
// dB_t = G_t, and column j of dA_t = G_t H_{t-1}^T, dA[r][j] = sum_c G[r][c]
// H_{t-1}[j][c]: the other columns of G_t come from the lane's three other
// threads (column j ^ d from the thread j ^ d), the matching elements
// H_{t-1}[j][j ^ d] from row j of the stage's H tile. offA[q]: row q of the
// block; offC[r]: element j of row r; offR[d]: element j ^ d of row j.
__device__ __forceinline__ void bwd_step(const unsigned char* As, const unsigned char* Hs,
                                         const unsigned char* Ds, unsigned char* OA,
                                         unsigned char* OB, int i, const int (&offA)[4],
                                         const int (&offC)[4], const int (&offR)[4],
                                         float (&g)[4]) {
  const int base = i * 512;
  float4 a[4];  // rows of A_{t+1}
#pragma unroll
  for (int q = 0; q < 4; ++q) a[q] = lds<float4>(As, base + offA[q]);
  float hr[4];  // H_{t-1}[j][j ^ d]
#pragma unroll
  for (int d = 0; d < 4; ++d) hr[d] = lds<float>(Hs, base + offR[d]);
  float gn[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float dh = lds<float>(Ds, base + offC[r]);
    gn[r] = fmaf(comp(a[3], r), g[3],
                 fmaf(comp(a[2], r), g[2], fmaf(comp(a[1], r), g[1], fmaf(comp(a[0], r), g[0], dh))));
  }
  float da[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    g[r] = gn[r];
    sts<float>(OB, base + offC[r], gn[r]);  // dB_t = G_t
    da[r] = gn[r] * hr[0];
  }
#pragma unroll
  for (int d = 1; d < 4; ++d)
#pragma unroll
    for (int r = 0; r < 4; ++r) da[r] = fmaf(__shfl_xor_sync(kFull, gn[r], d), hr[d], da[r]);
#pragma unroll
  for (int r = 0; r < 4; ++r) sts<float>(OA, base + offC[r], da[r]);
}

__global__ void __launch_bounds__(32) affine44_ring_bwd(const __grid_constant__ RingParams p) {
  constexpr int NS = kRingStagesBwd;
  extern __shared__ unsigned char ring_smem[];
  __shared__ unsigned long long bars[NS + 1];
  const int lane = threadIdx.x, l = lane >> 2, j = lane & 3;
  const int b = blockIdx.x / p.gpb;
  const int n0 = (blockIdx.x % p.gpb) * kRingLanes;
  const int64_t n = n0 + l;
  unsigned char* stage0 = ring_base(ring_smem);
  unsigned char* out0 = stage0 + (size_t)NS * 3 * kTile;
  const int nch = p.nchunks;
  // u-th chunk in walk order is chunk nch - 1 - u; its tiles: A from step t0 + 1
  // (A_{t+1} of every step t of the chunk; past T the fill is 0), H from step
  // t0 - 1 (H_{t-1}; step -1 is outside the tensor: the warp writes h0 there),
  // dH from step t0
  auto issue = [&](int u) {
    const int s = u % NS;
    unsigned char* st = stage0 + (size_t)s * 3 * kTile;
    const int t0 = (nch - 1 - u) * kRingLC;
    mbar_expect_tx(&bars[s], 3 * kTile);
    tma_load_4d(st, &p.in[0], 0, n0, t0 + 1, b, &bars[s]);
    tma_load_4d(st + kTile, &p.in[1], 0, n0, t0 - 1, b, &bars[s]);
    tma_load_4d(st + 2 * kTile, &p.in[2], 0, n0, t0, b, &bars[s]);
  };
  if (lane == 0) {
    for (int s = 0; s <= NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    for (int u = 0; u < NS && u < nch; ++u) issue(u);
  }
  __syncwarp();

  const int sl = (l >> 1) & 3;
  int offA[4], offC[4], offR[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    offA[q] = l * 64 + ((q ^ sl) << 4);
    offC[q] = offA[q] + 4 * j;
    offR[q] = l * 64 + ((j ^ sl) << 4) + 4 * (j ^ q);
  }
  float g[4] = {0.f, 0.f, 0.f, 0.f};  // column j of G_{t+1}

  for (int u = 0; u < nch; ++u) {
    const int s = u % NS;
    unsigned long long* bar = (p.test_stall && blockIdx.x == 0 && u == 1) ? &bars[NS] : &bars[s];
    if (!mbar_wait(bar, (unsigned)((u / NS) & 1), p.wait_limit_ns)) {
      if (lane == 0) {
        record_timeout(p, nch - 1 - u);
        drain<NS>(bars, u, (u + NS < nch ? u + NS : nch), p.wait_limit_ns);
      }
      return;
    }
    if (lane == 0) bulk_wait_read<1>();  // the stores of two chunks ago (dA, dB: one group)
    __syncwarp();
    const unsigned char* As = stage0 + (size_t)s * 3 * kTile;
    unsigned char* Hs = stage0 + (size_t)s * 3 * kTile + kTile;
    const unsigned char* Ds = Hs + kTile;
    unsigned char* OA = out0 + (size_t)(u & 1) * 2 * kTile;
    unsigned char* OB = OA + kTile;
    const int64_t t0 = (int64_t)(nch - 1 - u) * kRingLC;
    if (t0 == 0) {
      // H_{-1} = h0 (0 when absent): row j of this lane's block, read back
      // only by this thread
      float4 hz = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p.h0 && n < p.N) hz = __ldg(reinterpret_cast<const float4*>(p.h0 + ((int64_t)b * p.N + n) * 16) + j);
      sts<float4>(Hs, l * 64 + ((j ^ sl) << 4), hz);  // piece j of the block
    }
    const int steps = p.T - t0 < kRingLC ? (int)(p.T - t0) : kRingLC;
    if (steps == kRingLC) {
#pragma unroll
      for (int i = kRingLC - 1; i >= 0; --i) bwd_step(As, Hs, Ds, OA, OB, i, offA, offC, offR, g);
    } else {
      for (int i = steps - 1; i >= 0; --i) bwd_step(As, Hs, Ds, OA, OB, i, offA, offC, offR, g);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_4d(&p.out[0], 0, n0, (int)t0, b, OA);
      tma_store_4d(&p.out[1], 0, n0, (int)t0, b, OB);
      bulk_commit();
      if (u + NS < nch) issue(u + NS);
    }
  }
  // dh0 = A_0^T G_0 (column j)
  if (p.dh0 && n < p.N) {
    const float4* A0 = reinterpret_cast<const float4*>(p.A + ((int64_t)b * p.T * p.N + n) * 16);
    float4 a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) a[q] = __ldg(A0 + q);
    float* dh0 = p.dh0 + ((int64_t)b * p.N + n) * 16;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      dh0[r * 4 + j] = fmaf(comp(a[3], r), g[3],
                            fmaf(comp(a[2], r), g[2], fmaf(comp(a[1], r), g[1], comp(a[0], r) * g[0])));
  }
  if (lane == 0) bulk_wait_all();
}

size_t ring_smem_bytes(bool fwd) {
  return fwd ? (size_t)(kRingStagesFwd * 2 + 2) * kTile + 1024
             : (size_t)(kRingStagesBwd * 3 + 4) * kTile + 1024;
}

}  // namespace

bool affine_ring_fits(int64_t B, int64_t T, int64_t N, int k, int v) {
  return k == 4 && v == 4 && N >= kRingLanes && T >= kRingLC && T <= 0x7fffffffLL - 2 * kRingLC &&
         N <= 0x7fffffffLL && B <= 0x7fffffffLL && B * ((N + kRingLanes - 1) / kRingLanes) <= 0x7fffffffLL;
}

int64_t affine_ring_warps(int64_t B, int64_t N) { return B * ((N + kRingLanes - 1) / kRingLanes); }

cudaError_t launch_affine_ring(const AffineParams& a, int mode, cudaStream_t s) {
  RingParams p;
  memset(&p, 0, sizeof(p));
  const bool fwd = mode == MODE_FWD;
  const float* ins[3] = {a.A, fwd ? a.Bm : a.H, fwd ? nullptr : a.dH};
  float* outs[2] = {fwd ? a.out_H : a.dA, fwd ? nullptr : a.dB};
  for (int i = 0; i < (fwd ? 2 : 3); ++i)
    if (!encode_blocks_map(&p.in[i], ins[i], a.B, a.T, a.N, kRingLC)) return cudaErrorInvalidValue;
  for (int i = 0; i < (fwd ? 1 : 2); ++i)
    if (!encode_blocks_map(&p.out[i], outs[i], a.B, a.T, a.N, kRingLC)) return cudaErrorInvalidValue;
  p.A = a.A;
  p.h0 = a.h0;
  p.dh0 = a.dh0;
  p.B = a.B;
  p.T = a.T;
  p.N = a.N;
  p.gpb = (int)((a.N + kRingLanes - 1) / kRingLanes);
  p.nchunks = (int)((a.T + kRingLC - 1) / kRingLC);
  p.hdr = a.hdr;
  p.wait_limit_ns = a.wait_limit_ns;
  p.test_stall = a.test_stall;
  const size_t smem = ring_smem_bytes(fwd);
  const int64_t grid = a.B * p.gpb;
  if (fwd) {
    cudaError_t e = cudaFuncSetAttribute(affine44_ring_fwd,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    affine44_ring_fwd<<<(unsigned)grid, 32, smem, s>>>(p);
  } else {
    cudaError_t e = cudaFuncSetAttribute(affine44_ring_bwd,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    affine44_ring_bwd<<<(unsigned)grid, 32, smem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace scan
