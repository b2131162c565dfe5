/*
 * libscan.h -- C ABI of libscan, the GB300 (sm_103a) associative affine scan.
 *
 * The library computes the first-order affine recurrence
 *
 *     h_t = A_t h_{t-1} + B_t
 *
 * forward and backward on one GPU, in three forms:
 *   - scalar, channel-wise: h[t] = a[t] * h[t-1] + x[t] over [B, C, T], with
 *     packed variable-length sequences (cu_seqlens), resets (a_t = 0), a
 *     nonzero initial state and two opposite-direction branches;
 *   - block matrix: A_t is k x k and B_t, h_t are k x v;
 *   - log space: the scalar recurrence carried as l_t = log h_t.
 *
 * Sources (page titles and sections of the pages that define the operation):
 *   [TSK]  "Triton scan kernels" (minGRU docs): One associative-scan family
 *          (the recurrence, its monoid and the four scan ops), Kernel design
 *          ((b, n) lanes, channel tiles, (k, v) blocks), The TF32 / IEEE
 *          precision guard (envelope k, v in {1, 2, 4, 8, 16}), Autograd
 *          integration and the reversed-scan backward.
 *   [AST]  "associative_scan_triton" README: quick start (scan_causal,
 *          scan_bidirectional_branched, cu_seqlens), how it works (chunked
 *          scan, no cross-document leakage, backward by a reverse scan on
 *          shifted gates with d_gates = shifted_states * d_tokens).
 *   [GDN]  "Operations & Triton Kernels" (HyMo): The chunked GDN algorithm;
 *          Mathematical Derivation of the Reverse-Time Backward Pass.
 *   [RGA]  "Our RG-LRU GPU audit": Strengthened fused path (resets, nonzero
 *          initial state and its gradient, partial final chunks), Exact real
 *          chunk algebra (h_out = P h_in + Q).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers to contiguous row-major arrays;
 *     scalars are passed by value. The caller owns every buffer. The library
 *     never allocates device memory and never synchronises the stream except
 *     in scan_get_device_status().
 *   - Every call is asynchronous on `stream`; it returns after validating its
 *     arguments on the host and enqueueing its kernel(s). No exception crosses
 *     the ABI and there is no fallback: an input outside what the kernels
 *     support returns an error status and computes nothing.
 *   - Time index t is 0-based and h_{-1} = h0 (zero when h0 is NULL).
 *   - Accumulation is always fp32. `a`, `x`, `da`, `dx` may be fp32 or bf16
 *     (scan_dtype); h, h0, dh, dh0 are always fp32 ([TSK] Kernel design:
 *     "Accumulation is fp32 regardless of input dtype").
 *   - Dense layout: a, x, h, dh, da, dx are [B, C, T]; h0, dh0 are [B, C].
 *     Packed layout (cu_seqlens != NULL): B must be 1, tensors are [C, T]
 *     with T the total packed length, cu_seqlens is a device int32 array of
 *     n_seqs + 1 non-decreasing offsets from 0 to T ([AST] quick start,
 *     flash-attn convention), h0/dh0 are [n_seqs, C]. Empty sequences are
 *     allowed; their dh0 rows are written as 0.
 *   - A reset is simply a_t = 0: it erases the prefix ([RGA] Exact real chunk
 *     algebra). No separate reset mask exists.
 *   - Workspace: a device buffer of scan_workspace_bytes() bytes that the
 *     caller allocates once and zeroes once with scan_workspace_init(). After
 *     that it may be reused by any number of calls on one stream without
 *     clearing; calls that run concurrently on the GPU need separate
 *     workspaces. It also holds the sticky device status word read by
 *     scan_get_device_status().
 *   - Scalar and log forms accept any base pointer; 16-byte aligned fp32
 *     tensors and 8-byte aligned bf16 tensors (torch allocations are) take
 *     the vectorised path. The block form needs 16-byte aligned tensors.
 */
#ifndef LIBSCAN_H
#define LIBSCAN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LIBSCAN_VERSION 1

typedef enum scan_status {
  SCAN_OK = 0,
  SCAN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum, malformed host cu_seqlens */
  SCAN_ERR_UNSUPPORTED = 2, /* outside the kernels' envelope (e.g. k, v not in {1,2,4,8,16}) */
  SCAN_ERR_ALIGNMENT = 3,   /* affine tensors must be 16-byte aligned */
  SCAN_ERR_WORKSPACE = 4,   /* workspace missing or smaller than scan_workspace_bytes() */
  SCAN_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
  SCAN_ERR_TIMEOUT = 6,     /* device: a look-back wait ran past opts.wait_limit_s */
  SCAN_ERR_SEQLENS = 7      /* device: cu_seqlens not 0 = cu[0] <= ... <= cu[n] = T */
} scan_status;

typedef enum scan_dtype {
  SCAN_F32 = 0,
  SCAN_BF16 = 1
} scan_dtype;

/* How T is split across thread blocks. STATIONARY: a block walks a row
 * group in order with the running state in registers ([TSK] Kernel design;
 * [RGA] state-stationary serial path); long rows may be cut into a few
 * segments, each block waiting once for the end state of the previous
 * segment. LOOKBACK: T is cut into chunks handled by independent blocks; each
 * block publishes its chunk summary (P, Q) ([RGA] Exact real chunk algebra)
 * and reads its predecessors' summaries (decoupled look-back). STREAM: a
 * persistent grid sized by occupancy; each warp walks a contiguous share of
 * whole rows with the running state in registers, its chunks arriving in a
 * ring of shared-memory stages by 2-D tensor copies (TMA) several chunks
 * ahead, and leaving through tensor stores; needs every tensor 16-byte
 * aligned and at least 64 elements (else it runs as STATIONARY). AUTO picks
 * per shape. */
typedef enum scan_variant {
  SCAN_VARIANT_AUTO = 0,
  SCAN_VARIANT_STATIONARY = 1,
  SCAN_VARIANT_LOOKBACK = 2,
  SCAN_VARIANT_STREAM = 3
} scan_variant;

typedef enum scan_op {
  SCAN_OP_FWD = 0,
  SCAN_OP_BWD = 1,
  SCAN_OP_BIDIR_FWD = 2,
  SCAN_OP_BIDIR_BWD = 3,
  SCAN_OP_LOG_FWD = 4,
  SCAN_OP_AFFINE_FWD = 5,
  SCAN_OP_AFFINE_BWD = 6,
  SCAN_OP_LOG_BWD = 7
} scan_op;

/* Optional tuning and test controls; pass NULL for the defaults (all zero). */
typedef struct scan_opts {
  int32_t variant;       /* scan_variant; 0 = AUTO */
  int32_t chunk;         /* scalar/log: elements of T per block row, one of 128, 256, 512;
                            affine: time steps per block, one of 64, 128, 256; 0 = planner */
  int32_t rows_per_cta;  /* scalar/log: rows (channels) per block, 1..8 (blocks of 32 x
                            rows_per_cta threads); 0 = planner */
  int32_t test_stall;    /* test hook: 1 makes one look-back wait on a summary that is
                            never published, so the wait limit expires (SCAN_ERR_TIMEOUT) */
  double wait_limit_s;   /* bound on every look-back wait; <= 0 means 1.0 second */
  const int32_t* cu_seqlens_host; /* optional host copy of cu_seqlens, validated before launch */
  int32_t segments;      /* stationary: segments each row is cut into (>= 1); 0 = planner */
  int32_t stages;        /* stream: chunks in flight per warp, 2..16; 0 = planner */
} scan_opts;

/* Human-readable name of a status code (static string, never NULL). */
const char* scan_status_string(scan_status status);

/* LIBSCAN_VERSION of the loaded library. */
int32_t scan_version(void);

/* Bytes of workspace a call of `op` with these sizes needs under `opts`
 * (NULL = defaults). Scalar/log ops: (B, C, T) as in the call, k = v = 0.
 * Affine ops: B = batch, C = N (state blocks), T = time, and k, v.
 * Returns 0 for arguments the call itself would reject. */
size_t scan_workspace_bytes(scan_op op, int64_t B, int64_t C, int64_t T,
                            int32_t k, int32_t v, const scan_opts* opts);

/* Zero a freshly allocated workspace (asynchronous on `stream`). */
scan_status scan_workspace_init(void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/* Synchronise `stream`, read the workspace's sticky device status
 * (SCAN_ERR_TIMEOUT, SCAN_ERR_SEQLENS or SCAN_OK), reset it to SCAN_OK and
 * return it. */
scan_status scan_get_device_status(void* workspace, cudaStream_t stream);

/* Scalar forward ([AST] quick start, scan_causal; [TSK] linear_scan):
 *   reverse == 0: h_t = a_t h_{t-1} + x_t, h_{-1} = h0;
 *   reverse != 0: h_t = a_t h_{t+1} + x_t, h_T = h0 (per row or sequence).
 * a, x: [B,C,T] or packed [C,T] of `dt`; h0: nullable fp32 [B,C] or
 * [n_seqs,C]; h: fp32 output. */
scan_status scan_fwd(const void* a, const void* x, const float* h0,
                     const int32_t* cu_seqlens, int32_t n_seqs, float* h,
                     int64_t B, int64_t C, int64_t T, scan_dtype dt,
                     int32_t reverse, const scan_opts* opts, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream);

/* Scalar backward of L = sum_t <dh_t, h_t> ([AST] how it works: d_tokens by a
 * reverse scan on shifted gates, d_gates = shifted_states * d_tokens):
 *   g_t = dh_t + a_{t+1} g_{t+1} (a_{t+1} = 0 past the sequence end),
 *   dx_t = g_t, da_t = g_t h_{t-1} (h_{-1} = h0), dh0 = a_0 g_0
 * (mirrored when reverse != 0). `h` is the forward output, used as the
 * shifted state so no forward state is recomputed or stored ([TSK]
 * Autograd integration: the backward reads only the forward's inputs and
 * outputs). h0 is needed for da at a sequence start (nullable = 0). da, dx
 * have dtype `dt`; dh0 is a nullable fp32 output. */
scan_status scan_bwd(const void* a, const float* h, const float* dh,
                     const float* h0, const int32_t* cu_seqlens, int32_t n_seqs,
                     void* da, void* dx, float* dh0, int64_t B, int64_t C,
                     int64_t T, scan_dtype dt, int32_t reverse,
                     const scan_opts* opts, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream);

/* Two independent branches in one launch ([AST] quick start,
 * scan_bidirectional_branched): branch f is causal over (af, xf), branch r
 * runs from each sequence's end over (ar, xr). Same result as scan_fwd with
 * reverse = 0 and reverse = 1; the outputs are separate, not summed. */
scan_status scan_bidir_fwd(const void* af, const void* xf, const void* ar,
                           const void* xr, const float* h0f, const float* h0r,
                           const int32_t* cu_seqlens, int32_t n_seqs,
                           float* hf, float* hr, int64_t B, int64_t C,
                           int64_t T, scan_dtype dt, const scan_opts* opts,
                           void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* Backward of both branches in one launch; equal to scan_bwd with
 * reverse = 0 on branch f and reverse = 1 on branch r. */
scan_status scan_bidir_bwd(const void* af, const float* hf, const float* dhf,
                           const float* h0f, const void* ar, const float* hr,
                           const float* dhr, const float* h0r,
                           const int32_t* cu_seqlens, int32_t n_seqs,
                           void* daf, void* dxf, float* dh0f, void* dar,
                           void* dxr, float* dh0r, int64_t B, int64_t C,
                           int64_t T, scan_dtype dt, const scan_opts* opts,
                           void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* Log-space forward ([TSK] One associative-scan family, parallel_scan_log):
 *   l_t = log(exp(l_{t-1} + log_a_t) + exp(log_x_t)), l_{-1} = log_h0
 *   (-inf when log_h0 is NULL), output h_t = exp(l_t) in linear space.
 * log_a may be -inf (a reset). All fp32; layouts as scan_fwd. */
scan_status scan_log_fwd(const float* log_a, const float* log_x,
                         const float* log_h0, const int32_t* cu_seqlens,
                         int32_t n_seqs, float* h, int64_t B, int64_t C,
                         int64_t T, int32_t reverse, const scan_opts* opts,
                         void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* Log-space backward of L = sum_t dh_t h_t with h = scan_log_fwd(...). The
 * adjoint is the linear one on a = exp(log_a), x = exp(log_x)
 * ([TSK] One associative-scan family; the chain rule through exp):
 *   g_t = dh_t + a_{t+1} g_{t+1} (a_{t+1} = 0 past a sequence end),
 *   dlog_x_t = g_t x_t, dlog_a_t = g_t a_t h_{t-1} (h_{-1} = exp(log_h0)),
 *   dlog_h0 = a_0 g_0 exp(log_h0) per row or sequence (0 without log_h0).
 * reverse mirrors the shifts as scan_bwd does. Inputs: log_a, log_x as given
 * to scan_log_fwd, h its output, dh fp32; all outputs fp32 in the same
 * layouts; dlog_h0 nullable. Runs STATIONARY or LOOKBACK (a STREAM request
 * runs STATIONARY). */
scan_status scan_log_bwd(const float* log_a, const float* log_x, const float* h,
                         const float* dh, const float* log_h0,
                         const int32_t* cu_seqlens, int32_t n_seqs,
                         float* dlog_a, float* dlog_x, float* dlog_h0, int64_t B,
                         int64_t C, int64_t T, int32_t reverse,
                         const scan_opts* opts, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/* Block-matrix forward ([TSK] One associative-scan family, matrix_affine_scan;
 * Kernel design): H_t = A_t H_{t-1} + B_t per (b, n) lane, H_{-1} = h0.
 * A: [B,T,N,k,k], Bm and H: [B,T,N,k,v], h0: nullable [B,N,k,v]; row-major
 * matrices; fp32, 16-byte aligned (else SCAN_ERR_ALIGNMENT). Supported
 * (k, v): k and v each in {1, 2, 4, 8, 16} ([TSK] Conformance envelope);
 * others return SCAN_ERR_UNSUPPORTED. (4, 4) and (2, 2) run a kernel that
 * keeps whole blocks in registers, every other shape one that streams A. */
scan_status affine_scan_fwd(const float* A, const float* Bm, const float* h0,
                            float* H, int64_t B, int64_t T, int64_t N,
                            int32_t k, int32_t v, const scan_opts* opts,
                            void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* Block-matrix backward of L = sum_t <dH_t, H_t> ([TSK] Autograd integration
 * and the reversed-scan backward): G_t = dH_t + A_{t+1}^T G_{t+1},
 * dB_t = G_t, dA_t = G_t H_{t-1}^T (H_{-1} = h0), dh0 = A_0^T G_0.
 * H is the forward output; dh0 is nullable. Same envelope as the forward. */
scan_status affine_scan_bwd(const float* A, const float* H, const float* dH,
                            const float* h0, float* dA, float* dB, float* dh0,
                            int64_t B, int64_t T, int64_t N, int32_t k,
                            int32_t v, const scan_opts* opts, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/* Coefficient prefix of the block scan ([TSK] One associative-scan family:
 * matrix_affine_scan composes the pairs (A, B) and returns the composed
 * coefficient as well): Abar_t = A_t A_{t-1} ... A_0 per (b, n) lane, i.e. the
 * block scan with v = k, B_t = 0 and h0 = I. A, Abar: [B,T,N,k,k] fp32,
 * 16-byte aligned; k in {1, 2, 4, 8, 16}; workspace as affine_scan_fwd with
 * v = k. */
scan_status affine_prefix_fwd(const float* A, float* Abar, int64_t B, int64_t T,
                              int64_t N, int32_t k, const scan_opts* opts,
                              void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/* Backward of L = sum_t <dAbar_t, Abar_t>: G_t = dAbar_t + A_{t+1}^T G_{t+1},
 * dA_t = G_t Abar_{t-1}^T (Abar_{-1} = I). Abar is affine_prefix_fwd's output.
 * accumulate != 0 adds into dA (so a dA already written by affine_scan_bwd
 * receives both gradient terms); otherwise dA is overwritten. */
scan_status affine_prefix_bwd(const float* A, const float* Abar,
                              const float* dAbar, float* dA, int32_t accumulate,
                              int64_t B, int64_t T, int64_t N, int32_t k,
                              const scan_opts* opts, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* Scalar-gated outer-product state ([GDN] The chunked GDN algorithm), per
 * (batch, head):  h_t = alpha_t h_{t-1} + b_t v_t^T (S x D),  h_{-1} = h0,
 *                 o_t = h_t^T c_t (a D-vector).
 * Layouts (fp32, T-major within a head): alpha [B,H,T]; b, c [B,H,T,S];
 * v, o [B,H,T,D]; h0 nullable [B,H,S,D] (0 when NULL). S, D in {16, 32}
 * (else SCAN_ERR_UNSUPPORTED); b, c, v, o, h0, ckpt 16-byte aligned (else
 * SCAN_ERR_ALIGNMENT). ckpt (nullable): gdn_checkpoint_bytes() bytes, filled
 * with the state before every 32nd step, [B,H,ceil(T/32),S,D]; the backward
 * starts from it. Computed in 64-step chunks run in parallel, from the state
 * between chunks carried by a short serial pass per head.
 * workspace: gdn_workspace_bytes() bytes of device memory, 16-byte aligned,
 * owned by the caller (else SCAN_ERR_WORKSPACE); no state is kept in it
 * between calls. Asynchronous on `stream`. */
size_t gdn_checkpoint_bytes(int64_t B, int64_t H, int64_t T, int64_t S,
                            int64_t D);
size_t gdn_workspace_bytes(int64_t B, int64_t H, int64_t T, int64_t S,
                           int64_t D);
scan_status gdn_fwd(const float* alpha, const float* b, const float* v,
                    const float* c, const float* h0, float* o, float* ckpt,
                    int64_t B, int64_t H, int64_t T, int64_t S, int64_t D,
                    void* workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/* Its backward for L = sum_t <dout_t, o_t> ([GDN] Mathematical Derivation of
 * the Reverse-Time Backward Pass, with alpha itself as the gate input):
 *   dh_t = c_t dout_t^T + alpha_{t+1} dh_{t+1},   dc_t = h_t dout_t,
 *   dv_t = dh_t^T b_t,  db_t = dh_t v_t,  dalpha_t = <dh_t, h_{t-1}>,
 *   dh0 = alpha_0 dh_0 (nullable).
 * Computed chunk by chunk over T ([GDN] The chunked GDN algorithm): within a
 * 32-step chunk the products above become small matrix products; only the
 * adjoint of the state between chunks runs serially. ckpt is the forward's
 * checkpoint buffer (for the same inputs and h0); no state is stored besides
 * it. workspace: as for gdn_fwd. Outputs in the layouts of the corresponding
 * inputs. */
scan_status gdn_bwd(const float* alpha, const float* b, const float* v,
                    const float* c, const float* ckpt, const float* dout,
                    float* dalpha, float* db, float* dv, float* dc, float* dh0,
                    int64_t B, int64_t H, int64_t T, int64_t S, int64_t D,
                    void* workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/* RG-LRU gate preparation fused in front of the scalar scan ("Our RG-LRU GPU
 * audit", Strengthened fused path: the recurrent input, two gate logits,
 * a_param, optional segment_pos and initial state, with the gate activations,
 * log_a, transition, square-root multiplier and write formed in registers and
 * never stored; Exact real chunk algebra: a reset is a_t = 0 with the
 * canonical write). The gate formulas are the method's own (the pages name
 * these tensors but do not print them):
 *   r_t = sigmoid(gate_a_t), i_t = sigmoid(gate_x_t),
 *   log_a_t = 8 r_t log(sigmoid(a_param[c])), a_t = exp(log_a_t),
 *   write_t = sqrt(1 - a_t^2) i_t x_t;
 *   where segment_pos[b, t] == 0 (a reset): a_t = 0, write_t = i_t x_t;
 *   h_t = a_t h_{t-1} + write_t, h_{-1} = h0 (zero when h0 is NULL).
 *   x, gate_a, gate_x: [B, C, T] of dtype dt (SCAN_F32, or SCAN_BF16: the
 *     page's BF16 boundaries, read into fp32 registers), T contiguous (the
 *     scalar scan's dense layout); h: fp32 [B, C, T] (the state is carried in
 *     fp32 either way); a_param: fp32 [C]; segment_pos: int32 [B, T], shared
 *     by the channels of a batch row, or NULL (no resets); h0: fp32 [B, C] or
 *     NULL. All device pointers; any alignment (rows of T % 4 == 0 elements
 *     from pointers aligned to four elements take the vector path).
 * Returns SCAN_ERR_INVALID_ARG for negative sizes, a bad dtype or a NULL
 * required pointer,
 * SCAN_ERR_UNSUPPORTED for C > 2^31 - 1, SCAN_ERR_CUDA if the launch fails.
 * Asynchronous on `stream`; no workspace, no allocation. */
scan_status rglru_fwd(const void* x, const void* gate_a, const void* gate_x,
                      const float* a_param, const int32_t* segment_pos, const float* h0,
                      float* h, int64_t B, int64_t C, int64_t T, scan_dtype dt,
                      cudaStream_t stream);

/* Its backward for L = sum_t dh_t h_t, recomputing the gate terms from the
 * logits (the same page: backward recomputation of the pointwise terms, the
 * clipped square-root backward, partial a_param gradients followed by a
 * reduction): the adjoint g_t = dh_t + a_{t+1} g_{t+1} (a_T = 0), then
 *   dx_t = g_t m_t i_t, dgate_x_t = g_t m_t x_t i_t (1 - i_t)   (m = sqrt(1 - a^2)),
 *   dL/da_t = g_t h_{t-1} + g_t i_t x_t (d sqrt(u)/du) (-2 a_t), u = 1 - a_t^2,
 *     with d sqrt(u)/du taken at max(u, 1e-6) (the clip),
 *   dgate_a_t = a_t dL/da_t 8 log(sigmoid(a_param)) r_t (1 - r_t),
 *   da_param[c] = sigmoid(-a_param[c]) sum_{b,t} a_t dL/da_t 8 r_t,
 *   dh0 = a_0 g_0; a reset step has dgate_a = 0 and m = 1.
 *   h: the forward's output for the same inputs; dh: fp32 [B, C, T];
 *   dx, dgate_a, dgate_x: [B, C, T] of dtype dt (bf16 rounded to nearest from
 *   the fp32 results); da_param: fp32 [C], written (not
 *   accumulated), summed over b and t in a fixed order; dh0: [B, C] or NULL.
 * Errors as for rglru_fwd. Asynchronous on `stream`; no workspace. */
scan_status rglru_bwd(const void* x, const void* gate_a, const void* gate_x,
                      const float* a_param, const int32_t* segment_pos, const float* h0,
                      const float* h, const float* dh, void* dx, void* dgate_a,
                      void* dgate_x, float* da_param, float* dh0, int64_t B, int64_t C,
                      int64_t T, scan_dtype dt, cudaStream_t stream);

/* One training step of dense rows (scan_fwd then scan_bwd, reverse = 0) whose
 * inputs and results are in host memory ([AST] the scan and its reversed-scan
 * backward; the rows of [B,C,T] are independent, so cutting between rows is
 * exact). The B*C rows are cut into `pieces` pieces (0: 8; at most 64): each
 * piece's inputs are copied to the device buffers on one internal stream, the
 * piece is scanned forward and backward on `stream`, and its results are copied
 * back on a second internal stream, so the copies of neighbouring pieces run
 * under the scans and both copy directions run together. Results equal those
 * of scan_fwd and scan_bwd on the whole problem with the same variant, bit for
 * bit when T is a multiple of 4; otherwise a piece's rows start at another
 * 4-element memory phase, which moves the kernels' run boundaries and so the
 * rounding (within the forms' usual tolerance).
 * host: a, x (dt), dh [B,C,T] and h0 [B,C] (nullable) in; h [B,C,T] fp32, da,
 *       dx (dt) and dh0 [B,C] (nullable, with h0 and the device's h0/dh0 on
 *       the same footing) out. Page-locked host memory is needed for the
 *       copies to overlap (pageable memory works, without overlap).
 * dev:  device buffers of the same shapes, owned by the caller; their
 *       contents are overwritten.
 * Host and device pointers must all be given except h0/dh0 (else
 * SCAN_ERR_INVALID_ARG). opts: as for scan_fwd, except that the variant
 * defaults to SCAN_VARIANT_STATIONARY (a piece has fewer rows than the GPU has
 * warp slots). workspace: scan_workspace_bytes(SCAN_OP_BWD, 1, C', T, ...) for
 * the largest piece of C' = ceil(B*C / pieces) rows, shared by the pieces'
 * scans (they run in order on `stream`). The options and shape of the
 * largest piece (SCAN_ERR_INVALID_ARG / SCAN_ERR_UNSUPPORTED) and the
 * workspace (missing, not 16-byte aligned or too small: SCAN_ERR_WORKSPACE)
 * are checked before anything is queued; a CUDA error after that returns
 * SCAN_ERR_CUDA with `stream` made to wait for the copies already queued.
 * Asynchronous: on return the whole step is queued and `stream` waits for its
 * last copy; calls on one device are serialised on the host. */
typedef struct {
  const void* a;
  const void* x;
  const float* h0;
  const float* dh;
  float* h;
  void* da;
  void* dx;
  float* dh0;
} scan_host_io;
typedef struct {
  void* a;
  void* x;
  float* h0;
  float* dh;
  float* h;
  void* da;
  void* dx;
  float* dh0;
} scan_device_io;
scan_status scan_step_host(const scan_host_io* host, const scan_device_io* dev,
                           int64_t B, int64_t C, int64_t T, scan_dtype dt,
                           int32_t pieces, const scan_opts* opts,
                           void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* scan_copy modes. */
typedef enum scan_copy_mode {
  SCAN_COPY_VEC = 0, /* 128-bit streaming loads and stores, grid-stride */
  SCAN_COPY_TMA = 1  /* 32 KB 2-D tensor-copy tiles through a shared-memory ring */
} scan_copy_mode;

/* Copies `bytes` from src to dst on the device: the achievable read + write
 * bandwidth that the scan kernels' roofline fractions are reported against.
 * No counterpart in the source pages (they time their kernels alone): it
 * exists so that the ceiling is measured on the same GPU, launch path and
 * stream as the kernels it bounds, by copies written the way those kernels
 * move data (SCAN_COPY_VEC: the register path's 16-byte vector accesses;
 * SCAN_COPY_TMA: the stream variant's tensor copies).
 *   src, dst: device pointers, 16-byte aligned, not overlapping.
 *   bytes: a multiple of 16 (VEC) or of 128 (TMA); 0 does nothing.
 *   status: nullable device word; a TMA wait that expires (1 s) sets it to
 *     SCAN_ERR_TIMEOUT (the call itself has already returned).
 * Returns SCAN_ERR_INVALID_ARG for a bad mode, null pointer or size,
 * SCAN_ERR_ALIGNMENT for misaligned pointers, SCAN_ERR_CUDA if the launch or
 * the tensor-map encoding fails. Asynchronous on `stream`; allocates nothing. */
scan_status scan_copy(const void* src, void* dst, size_t bytes, int32_t mode, uint32_t* status,
                      cudaStream_t stream);

/* Bytes of the library's own scratch used by scan_fwd_noalloc (16 MiB). */
#define SCAN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* scan_fwd without a caller-provided workspace and without any allocation.
 * No counterpart in the source pages: it exists for callers that cannot
 * allocate device memory -- code running inside a memory-capped or
 * pre-partitioned arena, real-time paths that forbid allocation after
 * start-up, plugin hosts that hand over only the tensors they own. The
 * caller still passes a, x, h0, cu_seqlens and h exactly as for scan_fwd
 * (same layouts and meaning); the look-back chunk summaries go to a fixed
 * scratch array of SCAN_NOALLOC_SCRATCH_BYTES compiled into the library,
 * which every GPU that loads the library keeps until the process exits.
 *   - Limit: the call needs 256 + 16 * rows * chunks bytes (rows = B*C, or C
 *     when packed; chunks = ceil((T + 3) / 512) for T > 256). Larger problems
 *     return SCAN_ERR_WORKSPACE and compute nothing; use scan_fwd for them.
 *   - The first call on each device sets the scratch up: it looks up the
 *     array's device address (cudaGetSymbolAddress, which may load the
 *     library's device code) and writes nothing; the array is zero when the
 *     module loads. Make that first call before any stream capture on that
 *     device.
 *   - a, x, h (and h0, cu_seqlens) must be device memory of the current
 *     device, whose scratch the call uses; other pointers return
 *     SCAN_ERR_INVALID_ARG.
 *   - Every call on a device shares the same scratch and leaves its contents
 *     behind; the kernel resets what the next call needs. Calls whose kernels
 *     overlap on the GPU (different streams, or threads) race on it and give
 *     undefined results: serialise them.
 *   - Device-side findings (a malformed cu_seqlens, an expired wait) are kept
 *     in that scratch; scan_noalloc_device_status reads them back. Host-side
 *     checks return their status as usual. Never calls cudaMalloc, cudaFree
 *     or any allocating routine. */
scan_status scan_fwd_noalloc(const void* a, const void* x, const float* h0,
                             const int32_t* cu_seqlens, int32_t n_seqs, float* h,
                             int64_t B, int64_t C, int64_t T, scan_dtype dt,
                             int32_t reverse, cudaStream_t stream);

/* The sticky device status of the current device's scan_fwd_noalloc scratch,
 * read and cleared: scan_get_device_status (synchronises `stream`, reads the
 * status word, resets it to 0) applied to the library's own scratch, which
 * the caller has no pointer to. Returns SCAN_OK, the finding of a call since
 * the last read (SCAN_ERR_TIMEOUT for an expired look-back wait,
 * SCAN_ERR_SEQLENS for a malformed device cu_seqlens), or SCAN_ERR_CUDA
 * when the synchronisation or copies fail. Like scan_fwd_noalloc, it
 * allocates nothing; the copies are synchronous. */
scan_status scan_noalloc_device_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBSCAN_H */
