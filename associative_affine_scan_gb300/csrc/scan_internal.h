// scan_internal.h -- structures shared by libscan's translation units.
//
// Host planner (scan_api.cu) and kernels (scan_scalar_*.cu, scan_affine.cu)
// agree on these layouts; nothing here is part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/libscan.h"

namespace scan {

// MODE_LOGBWD: the backward of the log-space form, run as the linear adjoint
// on a = exp(log a) with the log-space chain rule applied to its outputs.
enum Mode { MODE_FWD = 0, MODE_BWD = 1, MODE_LOGBWD = 2 };
// Carry schemes. The first three are public (scan_variant); SEGMENTED is the
// stationary scheme with rows cut into segments, compiled separately so the
// plain stationary kernel keeps its register budget.
enum Variant { VAR_STATIONARY = 1, VAR_LOOKBACK = 2, VAR_STREAM = 3, VAR_SEGMENTED = 4 };

__host__ __device__ constexpr size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Stream variant: each warp walks whole rows through a ring of shared-memory
// stages, one chunk per stage, each input tile brought in by one 2-D tensor
// copy (TMA) with the 128-byte swizzle; outputs of interior chunks leave
// through swizzled tiles and tensor stores. A tensor is viewed as a flat
// [n / E, E] array of 128-byte rows (E = 128 / element size), so every tile
// starts on a 128-byte row: a chunk's first step is aligned to E elements of
// the flat tensor. Tiles are padded to 1024 bytes, the span of the swizzle.
constexpr int kMaxStages = 16;
__host__ __device__ constexpr int tma_row_elems(int elt) { return 128 / elt; }
__host__ __device__ constexpr size_t tma_tile_bytes(int J, int elt) {
  return (size_t)((128 * J * elt + 1023) / 1024 * 1024);
}
// input tiles of one stage: forward a, x; backward a, h, dh
__host__ __device__ constexpr size_t tma_stage_bytes(int mode, int J, int elt_a) {
  return mode == MODE_FWD ? 2 * tma_tile_bytes(J, elt_a)
                          : tma_tile_bytes(J, elt_a) + 2 * tma_tile_bytes(J, 4);
}
// output tiles of one buffer: forward h; backward dx, da
__host__ __device__ constexpr size_t tma_out_bytes(int mode, int J, int elt_a) {
  return mode == MODE_FWD ? tma_tile_bytes(J, 4) : 2 * tma_tile_bytes(J, elt_a);
}
// Dynamic shared memory of a stream block: packed offsets, mbarriers, 1 KB of
// alignment slack, then per warp ns stages and (with output tiles) two
// output buffers.
__host__ __device__ constexpr size_t tma_bar_bytes(int R) { return (size_t)R * kMaxStages * 8; }
__host__ __device__ constexpr size_t tma_warp_bytes(int mode, int J, int elt_a, int ns,
                                                    bool out_tiles) {
  return (size_t)ns * tma_stage_bytes(mode, J, elt_a) +
         (out_tiles ? 2 * tma_out_bytes(mode, J, elt_a) : 0);
}

// Workspace header, at offset 0 of every workspace. The look-back kernels take
// a tile ticket from `ticket_epoch` (low 32 bits) and read the launch epoch
// from its high 32 bits in the same atomic; the last block of a launch resets
// the ticket, advances the epoch and clears `done`, so no per-call memset is
// needed. `status` is the sticky device error (a scan_status value).
struct alignas(64) WsHeader {
  unsigned long long ticket_epoch;
  unsigned int done;
  unsigned int status;
  unsigned int info[4];  // where a wait expired: tile ticket, branch, row, scan index
  // two-branch stationary launches: row-group tickets per branch, and the
  // count of finished blocks (the last one resets all three)
  unsigned int branch_ticket[2];
  unsigned int branch_done;
  // the most record bytes any launch has used on this workspace since the
  // records were last cleared (see finish_lookback_launch)
  unsigned long long rec_bytes;
};
static_assert(sizeof(WsHeader) <= 256, "the header fits its 256 bytes");

constexpr size_t kWsHeaderBytes = 256;  // records start here

#ifdef __CUDACC__
// End of a launch that took tile tickets, run by thread 0 of the block that
// finished last (every other block has counted itself done after its work):
// clear the completion count, reset the ticket and advance the epoch.
// Record tags carry only the epoch's low 30 bits (tag = epoch * 4 + kind), so
// on one workspace a tag comes back every 2^30 launches. A record that no
// launch rewrote in between would then pass for a current one; so before the
// epoch whose tag bits wrap to zero, every record byte any launch has used
// since the last clear is zeroed (a zero word carries tag 0, which no record
// kind uses). This costs one pass over the records per 2^30 launches.
__device__ __forceinline__ void finish_lookback_launch(WsHeader* hdr, void* recs,
                                                       unsigned long long rec_bytes,
                                                       uint32_t epoch) {
  hdr->done = 0u;
  if (rec_bytes > hdr->rec_bytes) hdr->rec_bytes = rec_bytes;
  const uint32_t next = epoch + 1u;
  if ((next & 0x3fffffffu) == 0u) {
    const unsigned long long n = hdr->rec_bytes / 4;  // records are whole floats
    uint4* w16 = static_cast<uint4*>(recs);           // 16-byte aligned (after the header)
    const unsigned long long n16 = n / 4;
    for (unsigned long long i = 0; i < n16; ++i) w16[i] = make_uint4(0u, 0u, 0u, 0u);
    unsigned int* w4 = static_cast<unsigned int*>(recs);
    for (unsigned long long i = n16 * 4; i < n; ++i) w4[i] = 0u;
    hdr->rec_bytes = 0ull;
    __threadfence();
  }
  atomicExch(&hdr->ticket_epoch, ((unsigned long long)next) << 32);
  __threadfence();
}
#endif
// Packed offsets are staged in shared memory when n_seqs + 1 entries fit in
// this many; otherwise the kernels read cu_seqlens from global memory.
constexpr int kCuSmemEntries = 4096;

// One branch of a scalar scan launch.
struct BranchArgs {
  const void* a;     // gate a (dtype dt); forward and backward
  const void* x;     // forward: x (dtype dt); log-space backward: log x
  const float* h;    // backward: forward output h
  const float* dh;   // backward: upstream gradient
  const float* h0;   // nullable initial state ([B,C] dense, [n_seqs,C] packed); log h0 in
                     // the log-space backward
  float* out_h;      // forward output
  void* dx;          // backward outputs (dtype dt)
  void* da;
  float* dh0;        // nullable
  int dir;           // direction of the forward recurrence: +1 causal, -1 reverse
};

struct ScalarParams {
  BranchArgs br[2];
  const int32_t* cu;  // nullable packed offsets
  int n_seqs;
  int nbr;            // branches in this launch (1 or 2)
  int64_t rows;       // B*C dense, C packed
  int64_t T;          // row length
  int M;              // chunks per row along T
  int G;              // row groups (blocks along rows)
  int R;              // rows (warps) per block
  int64_t ntiles;     // look-back: M * G * nbr; segmented stationary: nseg * G * nbr
  int nseg;           // stationary: segments per row (1 = one block walks the whole row)
  int cps;            // stationary: chunks per segment
  int ns;             // stream: stages per warp
  int rpw;            // stream: rows (branch-major) per warp
  int tma_out;        // stream: interior chunks leave through tiles and tensor stores
  int64_t tile_hi;    // stream: flat elements [0, tile_hi) of every input are reachable by tiles
  unsigned long long* recs;  // look-back records: [nbr][rows][M] x 16 bytes
  unsigned long long rec_bytes;  // bytes of records this launch may use
  WsHeader* hdr;
  unsigned long long wait_limit_ns;
  int test_stall;
};

struct ScalarPlan {
  int variant;  // VAR_*
  int J;        // 128-element blocks per chunk (chunk = 128 J)
  int R;
  int M;
  int G;
  int nseg;     // stationary: segments per row
  int cps;      // stationary: chunks per segment
  bool vec;     // vectorised loads/stores
  int ns;       // stream: stages per warp
  bool tma_out; // stream: outputs through tiles and tensor stores
  size_t ws_bytes;
  size_t smem;
};

// Stream variant: the tensor maps of a launch, per branch (kernel parameter).
struct TmaMaps {
  CUtensorMap in[2][3];   // forward: a, x; backward: a, h, dh
  CUtensorMap out[2][2];  // forward: h; backward: dx, da
};

// Encodes the flat [n / E, E] view of a tensor of n elements of elt bytes, with
// tiles of 128 J elements and the 128-byte swizzle. False if the driver entry
// point is missing or refuses the map.
bool encode_tile_map(CUtensorMap* m, const void* ptr, int elt, int64_t n, int J);
bool encode_rows_map(CUtensorMap* m, const void* ptr, int64_t rows, int box_rows);
bool encode_blocks_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t N,
                       int box_steps);

// Launchers (one translation unit per mode/dtype family).
cudaError_t launch_scalar_fwd_f32(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s);
cudaError_t launch_scalar_fwd_bf16(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s);
cudaError_t launch_scalar_bwd_f32(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s);
cudaError_t launch_scalar_bwd_bf16(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s);
cudaError_t launch_log_fwd(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s);
cudaError_t launch_log_bwd(const ScalarParams& p, const ScalarPlan& pl, cudaStream_t s);

// Packed rows of the linear form (cu_seqlens), and dense bf16 rows of its
// backward, stationary, vectorised, chunks of 256 steps: the dedicated
// kernels of scan_packed.cu (mode MODE_FWD or MODE_BWD, elt = element size of
// a and x).
bool packed_applies(const ScalarParams& p, const ScalarPlan& pl, int mode, int elt);
cudaError_t launch_packed(const ScalarParams& p, const ScalarPlan& pl, int mode, int elt,
                          cudaStream_t s);

// Block-matrix affine scan.
struct AffineParams {
  const float* A;
  const float* Bm;
  const float* H;    // backward: forward output
  const float* dH;   // backward
  const float* h0;   // nullable; see flags
  float* out_H;      // forward output
  float* dA;
  float* dB;
  float* dh0;
  int64_t B, T, N;
  int k, v;
  int flags;         // AFF_* below
  int Lc;            // time steps per chunk
  int M;             // chunks along T
  int G;             // lane groups = B * ceil(N / 32)
  int64_t ntiles;
  float* recs;       // look-back records: [B*N][M] x record floats
  unsigned long long rec_bytes;  // bytes of records this launch may use
  WsHeader* hdr;
  unsigned long long wait_limit_ns;
  int test_stall;
};

// AffineParams.flags. The coefficient prefix Abar_t = A_t ... A_0 is the same
// scan with v = k, no injection and the identity as initial state; its
// gradient adds into the dA of the state's backward.
constexpr int AFF_ZERO_B = 1;   // Bm is absent: B_t = 0
constexpr int AFF_EYE_H0 = 2;   // h0 = I (k = v); h0 pointer unused
constexpr int AFF_ACC_DA = 4;   // backward adds into dA instead of writing it

struct AffinePlan {
  int variant;  // VAR_STATIONARY: the ring kernel (4 x 4 blocks); VAR_LOOKBACK otherwise
  int Lc;
  int M;
  int G;
  size_t ws_bytes;
};

// Floats per (lane, chunk) record for block shape (k, v); 0 if unsupported
// (k, v in {1, 2, 4, 8, 16} are supported).
int affine_record_floats(int k, int v);
int affine_sub_chunks();
// state blocks (lanes) per warp: 32 / max(k, v) column threads
int affine_lanes_per_block(int k, int v);

// Kernels for the shapes the register kernel does not cover, one launcher
// per k (mode: MODE_FWD or MODE_BWD).
cudaError_t launch_affine_generic_k1(const AffineParams& p, int mode, cudaStream_t s);
cudaError_t launch_affine_generic_k2(const AffineParams& p, int mode, cudaStream_t s);
cudaError_t launch_affine_generic_k4(const AffineParams& p, int mode, cudaStream_t s);
cudaError_t launch_affine_generic_k8(const AffineParams& p, int mode, cudaStream_t s);
cudaError_t launch_affine_generic_k16_fwd(const AffineParams& p, cudaStream_t s);
cudaError_t launch_affine_generic_k16_bwd(const AffineParams& p, cudaStream_t s);

// The 4 x 4 state-stationary kernels fed by a ring of tensor copies
// (scan_affine_ring.cu): shapes they take, warps they launch, launcher.
bool affine_ring_fits(int64_t B, int64_t T, int64_t N, int k, int v);
int64_t affine_ring_warps(int64_t B, int64_t N);
cudaError_t launch_affine_ring(const AffineParams& p, int mode, cudaStream_t s);

cudaError_t launch_affine_fwd(const AffineParams& p, const AffinePlan& pl, cudaStream_t s);
cudaError_t launch_affine_bwd(const AffineParams& p, const AffinePlan& pl, cudaStream_t s);

// Writes zeros to n floats (empty-input edge cases).
cudaError_t launch_fill_zero(float* p, int64_t n, cudaStream_t s);

// Status the planner gives dense rows of the scalar form with these options
// (every layout it may pick), without launching anything: SCAN_OK,
// SCAN_ERR_INVALID_ARG or SCAN_ERR_UNSUPPORTED.
scan_status scalar_plan_status(int64_t rows, int64_t T, int nbr, const scan_opts* opts);

}  // namespace scan
