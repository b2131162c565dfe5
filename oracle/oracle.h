/*
 * oracle.h -- sequential fp64 CPU oracle for the associative affine scan.
 *
 * TEST INFRASTRUCTURE ONLY. This code exists to check the CUDA library, not to
 * serve as a compute path. Only the test suite, the package smoke check and the
 * CPU-baseline leg of the benchmark may load it. It shares no code, header,
 * table or helper with the CUDA library, and it never calls it.
 *
 * Every routine is a plain, slow, left-to-right loop in double precision that
 * writes out the recurrence as the source pages define it:
 *
 *   "Triton scan kernels" (minGRU docs), section "One associative-scan family":
 *       h_t = A_t h_{t-1} + B_t, the scalar case being linear_scan (k = 1), the
 *       (k, v) block case matrix_affine_scan, and the log-space realisation
 *       parallel_scan_log.
 *   "associative_scan_triton" README, "quick start" and "how it works":
 *       h[t] = g[t] * h[t-1] + x[t] per channel, sequences packed with
 *       cu_seqlens (each scanned independently), two opposite-direction branches,
 *       and a backward that reverse-scans d_tokens on shifted gates and forms
 *       d_gates = shifted_states * d_tokens.
 *   "Our RG-LRU GPU audit", section "Exact real chunk algebra":
 *       a chunk summary h_out = P h_in + Q built left to right by
 *       P <- a_t P, Q <- a_t Q + b_t; a reset is a_t = 0.
 *
 * Layouts (all arrays contiguous, row-major):
 *   dense scalar : a, x, h, dh, da, dx are [B, C, T]; h0, dh0 are [B, C].
 *   varlen scalar: B must be 1; a, x, ... are [C, T] with T the packed length;
 *                  cu_seqlens is int32[n_seqs + 1] (0 = cu[0] <= ... <= cu[n_seqs] = T);
 *                  h0, dh0 are [n_seqs, C].
 *   affine       : A [B, T, N, k, k], Bm/H/dH/dB [B, T, N, k, v], h0/dh0 [B, N, k, v].
 * Time index t is 0-based and h_{-1} = h0 (zero when h0 is NULL). With
 * reverse != 0 a row (or segment) is scanned from its last element:
 *   h_t = a_t h_{t+1} + x_t, with h_{end} = h0.
 *
 * All functions return 0 on success and -1 on a malformed argument.
 */
#ifndef SCAN_ORACLE_H
#define SCAN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Scalar forward: h_t = a_t h_{t-1} + x_t per row / per segment. */
int oracle_scan_fwd(const double* a, const double* x, const double* h0,
                    const int32_t* cu_seqlens, int n_seqs, double* h,
                    int64_t B, int64_t C, int64_t T, int reverse);

/* Scalar backward of L = sum_t dh_t h_t. Recomputes its own fp64 forward states
 * from (a, x, h0). Writes da, dx (same layout as a) and, when dh0 != NULL, dh0. */
int oracle_scan_bwd(const double* a, const double* x, const double* h0,
                    const int32_t* cu_seqlens, int n_seqs, const double* dh,
                    double* da, double* dx, double* dh0,
                    int64_t B, int64_t C, int64_t T, int reverse);

/* Log-space forward: l_t = log(exp(l_{t-1} + log_a_t) + exp(log_x_t)),
 * l_{-1} = log_h0 (or -inf when log_h0 is NULL); writes h_t = exp(l_t). */
int oracle_scan_log_fwd(const double* log_a, const double* log_x,
                        const double* log_h0, const int32_t* cu_seqlens,
                        int n_seqs, double* h, int64_t B, int64_t C, int64_t T,
                        int reverse);

/* Log-space backward of L = sum_t dh_t h_t with respect to log_a, log_x and
 * log_h0 (chain rule through a = exp(log_a), x = exp(log_x), h0 = exp(log_h0)). */
int oracle_scan_log_bwd(const double* log_a, const double* log_x,
                        const double* log_h0, const int32_t* cu_seqlens,
                        int n_seqs, const double* dh, double* dlog_a,
                        double* dlog_x, double* dlog_h0,
                        int64_t B, int64_t C, int64_t T, int reverse);

/* Block-matrix forward: H_t = A_t H_{t-1} + B_t per (b, n) lane, H_{-1} = h0. */
int oracle_affine_fwd(const double* A, const double* Bm, const double* h0,
                      double* H, int64_t B, int64_t T, int64_t N, int k, int v);

/* Block-matrix backward of L = sum_t <dH_t, H_t>. Writes dA, dB and (when
 * non-NULL) dh0. Recomputes the forward states itself. */
int oracle_affine_bwd(const double* A, const double* Bm, const double* h0,
                      const double* dH, double* dA, double* dB, double* dh0,
                      int64_t B, int64_t T, int64_t N, int k, int v);

/* Scalar-gated outer-product state ("Operations & Triton Kernels" (HyMo),
 * The chunked GDN algorithm): per (batch, head)
 *   h_t = alpha_t h_{t-1} + b_t v_t^T   (S x D), h_{-1} = h0 (or 0)
 *   o_t = h_t^T c_t                      (D)
 * Layouts: alpha [B,H,T]; b, c [B,H,T,S]; v, o [B,H,T,D]; h0 [B,H,S,D]. */
int oracle_gdn_fwd(const double* alpha, const double* b, const double* v,
                   const double* c, const double* h0, double* o, int64_t B,
                   int64_t H, int64_t T, int64_t S, int64_t D);

/* Its backward for L = sum_t <do_t, o_t> (the same page, Mathematical
 * Derivation of the Reverse-Time Backward Pass), with alpha as the gate
 * input: dh_t = c_t do_t^T + alpha_{t+1} dh_{t+1}; dc_t = h_t do_t;
 * dv_t = dh_t^T b_t; db_t = dh_t v_t; dalpha_t = sum(dh_t * h_{t-1});
 * dh0 = alpha_0 dh_0. States from its own fp64 forward. */
int oracle_gdn_bwd(const double* alpha, const double* b, const double* v,
                   const double* c, const double* h0, const double* dout,
                   double* dalpha, double* db, double* dv, double* dc,
                   double* dh0, int64_t B, int64_t H, int64_t T, int64_t S,
                   int64_t D);

/* RG-LRU gate preparation in front of the scalar scan ("Our RG-LRU GPU audit",
 * Strengthened fused path: recurrent input x, two gate logits, a_param, an
 * optional segment_pos and initial state; gate activations, log_a, transition
 * a, square-root multiplier and write; Exact real chunk algebra: a reset is
 * a_t = 0 with the canonical reset write). The gate formulas are the method's
 * own; the pages name each of these tensors but do not print them:
 *   r_t = sigmoid(gate_a_t), i_t = sigmoid(gate_x_t),
 *   log_a_t = -8 softplus(-a_param[c]) r_t, a_t = exp(log_a_t),
 *   write_t = sqrt(1 - a_t^2) i_t x_t,
 *   where segment_pos[b, t] == 0 (a reset): a_t = 0 and write_t = i_t x_t;
 *   h_t = a_t h_{t-1} + write_t, h_{-1} = h0 (or 0).
 * Layouts: x, gate_a, gate_x, h [B, C, T]; a_param [C]; segment_pos int32
 * [B, T] (NULL: no resets); h0 [B, C]. */
int oracle_rglru_fwd(const double* x, const double* gate_a, const double* gate_x,
                     const double* a_param, const int32_t* segment_pos,
                     const double* h0, double* h, int64_t B, int64_t C, int64_t T);

/* Its backward for L = sum_t dh_t h_t: dx, dgate_a, dgate_x (layout of x),
 * da_param [C] (summed over B and T), dh0 [B, C] (when non-NULL). The
 * adjoint g_t = dh_t + a_{t+1} g_{t+1} (a_T = 0), then the chain rule through
 * the gate terms; the square root's derivative d sqrt(u) / du is taken at
 * max(u, 1e-6) (the clipped square-root backward), u = 1 - a_t^2. States
 * from its own fp64 forward. */
int oracle_rglru_bwd(const double* x, const double* gate_a, const double* gate_x,
                     const double* a_param, const int32_t* segment_pos,
                     const double* h0, const double* dh, double* dx,
                     double* dgate_a, double* dgate_x, double* da_param,
                     double* dh0, int64_t B, int64_t C, int64_t T);

/* Chunk summary of n consecutive scalar steps, built left to right
 * (P <- a_t P, Q <- a_t Q + x_t from P = 1, Q = 0). */
void oracle_chunk_summary(const double* a, const double* x, int64_t n,
                          double* P, double* Q);

/* Composition "apply (P1, Q1) then (P2, Q2)" = (P2 P1, P2 Q1 + Q2). */
void oracle_compose(double P1, double Q1, double P2, double Q2,
                    double* P, double* Q);

#ifdef __cplusplus
}
#endif

#endif /* SCAN_ORACLE_H */
