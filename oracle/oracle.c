/*
 * oracle.c -- sequential fp64 CPU oracle for the associative affine scan.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): loaded by the tests, the package
 * smoke check and the benchmark's CPU-baseline leg; never by the library.
 * Parity with it is pinned, independently of this file, by closed forms,
 * brute force on tiny inputs and invariants in tests/test_oracle_pins.py.
 *
 * Build: cc -O2 -ffp-contract=off -shared -fPIC oracle.c -lm
 * (-ffp-contract=off keeps a*b + c as two rounded operations on every host,
 * so x86-64 and aarch64 give the same bits.)
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* cu_seqlens follows the flash-attn convention named in the
 * "associative_scan_triton" README ("how it works"): non-decreasing offsets
 * from 0 to the packed length. Empty segments are allowed. */
static int check_segments(const int32_t* cu, int n_seqs, int64_t B, int64_t T) {
  if (!cu) return 0;
  if (B != 1 || n_seqs < 1) return -1;
  if (cu[0] != 0 || (int64_t)cu[n_seqs] != T) return -1;
  for (int i = 0; i < n_seqs; ++i)
    if (cu[i + 1] < cu[i]) return -1;
  return 0;
}

/* Segment s of a row: [beg, end). Dense rows are one segment [0, T). */
static void segment_bounds(const int32_t* cu, int s, int64_t T, int64_t* beg,
                           int64_t* end) {
  if (cu) {
    *beg = cu[s];
    *end = cu[s + 1];
  } else {
    *beg = 0;
    *end = T;
  }
}

/* Index of the initial state of segment s of row r: [B, C] dense, [n_seqs, C]
 * packed (B == 1 there, so the row is the channel). */
static int64_t h0_index(const int32_t* cu, int s, int64_t r, int64_t C) {
  return cu ? (int64_t)s * C + r : r;
}

/* "associative_scan_triton" README, quick start: h[t] = g[t] * h[t-1] + x[t],
 * each packed sequence scanned on its own; the reverse branch of
 * scan_bidirectional_branched runs the same recurrence from the segment end. */
int oracle_scan_fwd(const double* a, const double* x, const double* h0,
                    const int32_t* cu, int n_seqs, double* h, int64_t B,
                    int64_t C, int64_t T, int reverse) {
  if (!a || !x || !h || B < 0 || C < 0 || T < 0) return -1;
  if (check_segments(cu, n_seqs, B, T)) return -1;
  const int64_t rows = B * C;
  const int nseg = cu ? n_seqs : 1;
  for (int64_t r = 0; r < rows; ++r) {
    const double* ar = a + r * T;
    const double* xr = x + r * T;
    double* hr = h + r * T;
    for (int s = 0; s < nseg; ++s) {
      int64_t beg, end;
      segment_bounds(cu, s, T, &beg, &end);
      double state = h0 ? h0[h0_index(cu, s, r, C)] : 0.0;
      if (!reverse) {
        for (int64_t t = beg; t < end; ++t) {
          state = ar[t] * state + xr[t];
          hr[t] = state;
        }
      } else {
        for (int64_t t = end - 1; t >= beg; --t) {
          state = ar[t] * state + xr[t];
          hr[t] = state;
        }
      }
    }
  }
  return 0;
}

/* "associative_scan_triton" README, how it works: the backward computes
 * d_tokens by a reverse scan on shifted gates and d_gates = shifted_states *
 * d_tokens. For the causal branch the shifted gate of step t is a_{t+1} (zero
 * past the segment end, so no gradient leaks between packed sequences) and the
 * shifted state is h_{t-1} (h0 at the segment start); the reverse branch mirrors
 * both shifts. The initial-state gradient ("Our RG-LRU GPU audit", fused path:
 * "nonzero initial state and its gradient") is a_first * d_tokens_first. */
int oracle_scan_bwd(const double* a, const double* x, const double* h0,
                    const int32_t* cu, int n_seqs, const double* dh, double* da,
                    double* dx, double* dh0, int64_t B, int64_t C, int64_t T,
                    int reverse) {
  if (!a || !x || !dh || !da || !dx || B < 0 || C < 0 || T < 0) return -1;
  if (check_segments(cu, n_seqs, B, T)) return -1;
  const int64_t rows = B * C;
  const int nseg = cu ? n_seqs : 1;
  double* hs = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  if (!hs) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    const double* ar = a + r * T;
    const double* xr = x + r * T;
    const double* dhr = dh + r * T;
    double* dar = da + r * T;
    double* dxr = dx + r * T;
    for (int s = 0; s < nseg; ++s) {
      int64_t beg, end;
      segment_bounds(cu, s, T, &beg, &end);
      const double init = h0 ? h0[h0_index(cu, s, r, C)] : 0.0;
      double d_init = 0.0;
      if (!reverse) {
        double state = init;
        for (int64_t t = beg; t < end; ++t) {
          state = ar[t] * state + xr[t];
          hs[t] = state;
        }
        double g = 0.0;
        for (int64_t t = end - 1; t >= beg; --t) {
          const double shifted_gate = (t + 1 < end) ? ar[t + 1] : 0.0;
          g = dhr[t] + shifted_gate * g;
          dxr[t] = g;
          const double shifted_state = (t > beg) ? hs[t - 1] : init;
          dar[t] = shifted_state * g;
        }
        if (end > beg) d_init = ar[beg] * dxr[beg];
      } else {
        double state = init;
        for (int64_t t = end - 1; t >= beg; --t) {
          state = ar[t] * state + xr[t];
          hs[t] = state;
        }
        double g = 0.0;
        for (int64_t t = beg; t < end; ++t) {
          const double shifted_gate = (t - 1 >= beg) ? ar[t - 1] : 0.0;
          g = dhr[t] + shifted_gate * g;
          dxr[t] = g;
          const double shifted_state = (t + 1 < end) ? hs[t + 1] : init;
          dar[t] = shifted_state * g;
        }
        if (end > beg) d_init = ar[end - 1] * dxr[end - 1];
      }
      if (dh0) dh0[h0_index(cu, s, r, C)] = d_init;
    }
  }
  free(hs);
  return 0;
}

/* log(exp(u) + exp(w)) with the larger term factored out; -inf is the
 * additive identity (a zero term). */
static double log_add_exp(double u, double w) {
  if (u == -INFINITY) return w;
  if (w == -INFINITY) return u;
  const double m = u > w ? u : w;
  return m + log1p(exp(-fabs(u - w)));
}

/* "Triton scan kernels", One associative-scan family: parallel_scan_log is the
 * same recurrence carried in log space, writing h = exp(.) directly. Step by
 * step, h_t = a_t h_{t-1} + x_t with a_t = exp(log_a_t), x_t = exp(log_x_t)
 * reads l_t = log(exp(l_{t-1} + log_a_t) + exp(log_x_t)). */
int oracle_scan_log_fwd(const double* log_a, const double* log_x,
                        const double* log_h0, const int32_t* cu, int n_seqs,
                        double* h, int64_t B, int64_t C, int64_t T,
                        int reverse) {
  if (!log_a || !log_x || !h || B < 0 || C < 0 || T < 0) return -1;
  if (check_segments(cu, n_seqs, B, T)) return -1;
  const int64_t rows = B * C;
  const int nseg = cu ? n_seqs : 1;
  for (int64_t r = 0; r < rows; ++r) {
    const double* la = log_a + r * T;
    const double* lx = log_x + r * T;
    double* hr = h + r * T;
    for (int s = 0; s < nseg; ++s) {
      int64_t beg, end;
      segment_bounds(cu, s, T, &beg, &end);
      double l = log_h0 ? log_h0[h0_index(cu, s, r, C)] : -INFINITY;
      if (!reverse) {
        for (int64_t t = beg; t < end; ++t) {
          l = log_add_exp(l + la[t], lx[t]);
          hr[t] = exp(l);
        }
      } else {
        for (int64_t t = end - 1; t >= beg; --t) {
          l = log_add_exp(l + la[t], lx[t]);
          hr[t] = exp(l);
        }
      }
    }
  }
  return 0;
}

/* Gradient of the log-space scan by the chain rule through the linear adjoint:
 * d log_a_t = da_t a_t, d log_x_t = dx_t x_t, d log_h0 = dh0 h0. */
int oracle_scan_log_bwd(const double* log_a, const double* log_x,
                        const double* log_h0, const int32_t* cu, int n_seqs,
                        const double* dh, double* dlog_a, double* dlog_x,
                        double* dlog_h0, int64_t B, int64_t C, int64_t T,
                        int reverse) {
  if (!log_a || !log_x || !dh || !dlog_a || !dlog_x || B < 0 || C < 0 || T < 0)
    return -1;
  if (check_segments(cu, n_seqs, B, T)) return -1;
  const int64_t n = B * C * T;
  const int64_t nh0 = cu ? (int64_t)n_seqs * C : B * C;
  double* a = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* x = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* h0 = log_h0 ? (double*)malloc(sizeof(double) * (size_t)(nh0 > 0 ? nh0 : 1)) : NULL;
  double* dh0 = (double*)malloc(sizeof(double) * (size_t)(nh0 > 0 ? nh0 : 1));
  int rc = -1;
  if (!a || !x || !dh0 || (log_h0 && !h0)) goto done;
  for (int64_t i = 0; i < n; ++i) {
    a[i] = exp(log_a[i]);
    x[i] = exp(log_x[i]);
  }
  if (h0)
    for (int64_t i = 0; i < nh0; ++i) h0[i] = exp(log_h0[i]);
  rc = oracle_scan_bwd(a, x, h0, cu, n_seqs, dh, dlog_a, dlog_x, dh0, B, C, T,
                       reverse);
  if (rc) goto done;
  for (int64_t i = 0; i < n; ++i) {
    dlog_a[i] *= a[i];
    dlog_x[i] *= x[i];
  }
  if (dlog_h0)
    for (int64_t i = 0; i < nh0; ++i) dlog_h0[i] = h0 ? dh0[i] * h0[i] : 0.0;
done:
  free(a);
  free(x);
  free(h0);
  free(dh0);
  return rc;
}

/* "Triton scan kernels", One associative-scan family and Kernel design:
 * h_t = A_t h_{t-1} + B_t with A_t a k x k matrix and B_t a k x v injection,
 * one (b, n) lane walking T in order. Row-major matrices. */
int oracle_affine_fwd(const double* A, const double* Bm, const double* h0,
                      double* H, int64_t B, int64_t T, int64_t N, int k, int v) {
  if (!A || !Bm || !H || B < 0 || T < 0 || N < 0 || k < 1 || v < 1 || k > 64 ||
      v > 64)
    return -1;
  const int64_t kk = (int64_t)k * k, kv = (int64_t)k * v;
  double* state = (double*)malloc(sizeof(double) * (size_t)kv);
  double* next = (double*)malloc(sizeof(double) * (size_t)kv);
  if (!state || !next) {
    free(state);
    free(next);
    return -1;
  }
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t n = 0; n < N; ++n) {
      for (int64_t e = 0; e < kv; ++e)
        state[e] = h0 ? h0[(b * N + n) * kv + e] : 0.0;
      for (int64_t t = 0; t < T; ++t) {
        const int64_t blk = (b * T + t) * N + n;
        const double* At = A + blk * kk;
        const double* Bt = Bm + blk * kv;
        for (int i = 0; i < k; ++i) {
          for (int j = 0; j < v; ++j) {
            double acc = 0.0;
            for (int l = 0; l < k; ++l) acc += At[i * k + l] * state[l * v + j];
            next[i * v + j] = acc + Bt[i * v + j];
          }
        }
        memcpy(state, next, sizeof(double) * (size_t)kv);
        memcpy(H + blk * kv, state, sizeof(double) * (size_t)kv);
      }
    }
  }
  free(state);
  free(next);
  return 0;
}

/* "Triton scan kernels", Autograd integration and the reversed-scan backward:
 * reverse-scan the output gradients with A_{t+1}^T (G_t = dH_t + A_{t+1}^T
 * G_{t+1}), then dL/dB_t = G_t and dL/dA_t = G_t H_{t-1}^T from the forward
 * states (H_{-1} = h0); dL/dh0 = A_0^T G_0. */
int oracle_affine_bwd(const double* A, const double* Bm, const double* h0,
                      const double* dH, double* dA, double* dB, double* dh0,
                      int64_t B, int64_t T, int64_t N, int k, int v) {
  if (!A || !Bm || !dH || !dA || !dB || B < 0 || T < 0 || N < 0 || k < 1 ||
      v < 1 || k > 64 || v > 64)
    return -1;
  const int64_t kk = (int64_t)k * k, kv = (int64_t)k * v;
  double* hs = (double*)malloc(sizeof(double) * (size_t)((T > 0 ? T : 1) * kv));
  double* g = (double*)malloc(sizeof(double) * (size_t)kv);
  double* gnew = (double*)malloc(sizeof(double) * (size_t)kv);
  double* init = (double*)malloc(sizeof(double) * (size_t)kv);
  if (!hs || !g || !gnew || !init) {
    free(hs);
    free(g);
    free(gnew);
    free(init);
    return -1;
  }
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t n = 0; n < N; ++n) {
      for (int64_t e = 0; e < kv; ++e)
        init[e] = h0 ? h0[(b * N + n) * kv + e] : 0.0;
      /* forward states of this lane */
      for (int64_t t = 0; t < T; ++t) {
        const int64_t blk = (b * T + t) * N + n;
        const double* At = A + blk * kk;
        const double* Bt = Bm + blk * kv;
        const double* prev = t > 0 ? hs + (t - 1) * kv : init;
        for (int i = 0; i < k; ++i)
          for (int j = 0; j < v; ++j) {
            double acc = 0.0;
            for (int l = 0; l < k; ++l) acc += At[i * k + l] * prev[l * v + j];
            hs[t * kv + i * v + j] = acc + Bt[i * v + j];
          }
      }
      /* reverse adjoint scan */
      for (int64_t e = 0; e < kv; ++e) g[e] = 0.0;
      for (int64_t t = T - 1; t >= 0; --t) {
        const int64_t blk = (b * T + t) * N + n;
        const double* dHt = dH + blk * kv;
        for (int i = 0; i < k; ++i)
          for (int j = 0; j < v; ++j) {
            double acc = 0.0;
            if (t + 1 < T) {
              const double* An = A + ((b * T + t + 1) * N + n) * kk;
              for (int l = 0; l < k; ++l) acc += An[l * k + i] * g[l * v + j];
            }
            gnew[i * v + j] = dHt[i * v + j] + acc;
          }
        memcpy(g, gnew, sizeof(double) * (size_t)kv);
        memcpy(dB + blk * kv, g, sizeof(double) * (size_t)kv);
        const double* prev = t > 0 ? hs + (t - 1) * kv : init;
        double* dAt = dA + blk * kk;
        for (int i = 0; i < k; ++i)
          for (int l = 0; l < k; ++l) {
            double acc = 0.0;
            for (int j = 0; j < v; ++j) acc += g[i * v + j] * prev[l * v + j];
            dAt[i * k + l] = acc;
          }
      }
      if (dh0) {
        double* d = dh0 + (b * N + n) * kv;
        for (int i = 0; i < k; ++i)
          for (int j = 0; j < v; ++j) {
            double acc = 0.0;
            if (T > 0) {
              const double* A0 = A + ((b * T) * N + n) * kk;
              for (int l = 0; l < k; ++l) acc += A0[l * k + i] * g[l * v + j];
            }
            d[i * v + j] = acc;
          }
      }
    }
  }
  free(hs);
  free(g);
  free(gnew);
  free(init);
  return 0;
}

/* "Our RG-LRU GPU audit", Exact real chunk algebra: the summary of a chunk is
 * h_out = P h_in + Q, updated left to right by P <- a_t P, Q <- a_t Q + b_t. */
void oracle_chunk_summary(const double* a, const double* x, int64_t n,
                          double* P, double* Q) {
  double p = 1.0, q = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    p = a[t] * p;
    q = a[t] * q + x[t];
  }
  *P = p;
  *Q = q;
}

/* "Triton scan kernels", One associative-scan family: "apply (A1, B1) then
 * (A2, B2)" is the affine map h -> A2 (A1 h + B1) + B2 = (A2 A1) h + (A2 B1 + B2),
 * a monoid with identity (I, 0). Scalar case. */
void oracle_compose(double P1, double Q1, double P2, double Q2, double* P,
                    double* Q) {
  *P = P2 * P1;
  *Q = P2 * Q1 + Q2;
}

/* "Operations & Triton Kernels" (HyMo), The chunked GDN algorithm: the write
 * h_t = alpha_t h_{t-1} + b_t (outer) v_t and the read o_t = c_t . h_t, one
 * step after the other for every (batch, head). */
int oracle_gdn_fwd(const double* alpha, const double* b, const double* v,
                   const double* c, const double* h0, double* o, int64_t B,
                   int64_t H, int64_t T, int64_t S, int64_t D) {
  if (!alpha || !b || !v || !c || !o || B < 0 || H < 0 || T < 0 || S < 1 || D < 1)
    return -1;
  double* h = (double*)malloc(sizeof(double) * (size_t)(S * D));
  if (!h) return -1;
  for (int64_t bh = 0; bh < B * H; ++bh) {
    for (int64_t i = 0; i < S * D; ++i) h[i] = h0 ? h0[bh * S * D + i] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const int64_t st = bh * T + t;
      const double al = alpha[st];
      for (int64_t s = 0; s < S; ++s)
        for (int64_t d = 0; d < D; ++d)
          h[s * D + d] = al * h[s * D + d] + b[st * S + s] * v[st * D + d];
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t s = 0; s < S; ++s) acc += c[st * S + s] * h[s * D + d];
        o[st * D + d] = acc;
      }
    }
  }
  free(h);
  return 0;
}

/* The same page, Mathematical Derivation of the Reverse-Time Backward Pass,
 * with alpha itself as the gate input (its dalpha is the page's decay-gate
 * gradient before the chain rule into the gate's parameters). The forward
 * states are kept (this is the oracle: O(T S D) memory is fine). */
int oracle_gdn_bwd(const double* alpha, const double* b, const double* v,
                   const double* c, const double* h0, const double* dout,
                   double* dalpha, double* db, double* dv, double* dc,
                   double* dh0, int64_t B, int64_t H, int64_t T, int64_t S,
                   int64_t D) {
  if (!alpha || !b || !v || !c || !dout || !dalpha || !db || !dv || !dc || B < 0 ||
      H < 0 || T < 0 || S < 1 || D < 1)
    return -1;
  const int64_t SD = S * D;
  double* hs = (double*)malloc(sizeof(double) * (size_t)((T + 1) * SD));
  double* dh = (double*)malloc(sizeof(double) * (size_t)SD);
  if (!hs || !dh) {
    free(hs);
    free(dh);
    return -1;
  }
  for (int64_t bh = 0; bh < B * H; ++bh) {
    /* hs[0] = h_{-1}, hs[t + 1] = h_t */
    for (int64_t i = 0; i < SD; ++i) hs[i] = h0 ? h0[bh * SD + i] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const int64_t st = bh * T + t;
      for (int64_t s = 0; s < S; ++s)
        for (int64_t d = 0; d < D; ++d)
          hs[(t + 1) * SD + s * D + d] =
              alpha[st] * hs[t * SD + s * D + d] + b[st * S + s] * v[st * D + d];
    }
    for (int64_t i = 0; i < SD; ++i) dh[i] = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      const int64_t st = bh * T + t;
      const double* ht = hs + (t + 1) * SD;
      const double* hp = hs + t * SD;
      /* dh_t = c_t do_t^T + alpha_{t+1} dh_{t+1} */
      const double an = (t + 1 < T) ? alpha[st + 1] : 0.0;
      for (int64_t s = 0; s < S; ++s)
        for (int64_t d = 0; d < D; ++d)
          dh[s * D + d] = c[st * S + s] * dout[st * D + d] + an * dh[s * D + d];
      for (int64_t s = 0; s < S; ++s) {
        double acc_c = 0.0, acc_b = 0.0;
        for (int64_t d = 0; d < D; ++d) {
          acc_c += ht[s * D + d] * dout[st * D + d];
          acc_b += dh[s * D + d] * v[st * D + d];
        }
        dc[st * S + s] = acc_c;
        db[st * S + s] = acc_b;
      }
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t s = 0; s < S; ++s) acc += b[st * S + s] * dh[s * D + d];
        dv[st * D + d] = acc;
      }
      double acc_a = 0.0;
      for (int64_t i = 0; i < SD; ++i) acc_a += dh[i] * hp[i];
      dalpha[st] = acc_a;
    }
    if (dh0)
      for (int64_t i = 0; i < SD; ++i) dh0[bh * SD + i] = (T > 0 ? alpha[bh * T] : 0.0) * dh[i];
  }
  free(hs);
  free(dh);
  return 0;
}

/* "Our RG-LRU GPU audit", Strengthened fused path and Exact real chunk
 * algebra, with the method's own gate formulas (see oracle.h): the gate
 * terms of every step, then the scalar recurrence, left to right. */
#define RG_SCALE 8.0    /* log_a = -RG_SCALE softplus(-a_param) r */
#define RG_U_MIN 1e-6   /* the square root's derivative is taken at u >= RG_U_MIN */

static double rg_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* log(sigmoid(p)) = -softplus(-p), without overflow for large |p| */
static double rg_log_sigmoid(double p) { return p < 0.0 ? p - log1p(exp(p)) : -log1p(exp(-p)); }

int oracle_rglru_fwd(const double* x, const double* gate_a, const double* gate_x,
                     const double* a_param, const int32_t* segment_pos,
                     const double* h0, double* h, int64_t B, int64_t C, int64_t T) {
  if (!x || !gate_a || !gate_x || !a_param || !h || B < 0 || C < 0 || T < 0) return -1;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t c = 0; c < C; ++c) {
      const double ls = rg_log_sigmoid(a_param[c]);
      double state = h0 ? h0[b * C + c] : 0.0;
      for (int64_t t = 0; t < T; ++t) {
        const int64_t e = (b * C + c) * T + t;
        const double in_gate = rg_sigmoid(gate_x[e]);
        double a, write;
        if (segment_pos && segment_pos[b * T + t] == 0) {
          a = 0.0;
          write = in_gate * x[e];
        } else {
          const double log_a = RG_SCALE * rg_sigmoid(gate_a[e]) * ls;
          a = exp(log_a);
          write = sqrt(-expm1(2.0 * log_a)) * in_gate * x[e];
        }
        state = a * state + write;
        h[e] = state;
      }
    }
  return 0;
}

int oracle_rglru_bwd(const double* x, const double* gate_a, const double* gate_x,
                     const double* a_param, const int32_t* segment_pos,
                     const double* h0, const double* dh, double* dx,
                     double* dgate_a, double* dgate_x, double* da_param,
                     double* dh0, int64_t B, int64_t C, int64_t T) {
  if (!x || !gate_a || !gate_x || !a_param || !dh || !dx || !dgate_a || !dgate_x ||
      !da_param || B < 0 || C < 0 || T < 0)
    return -1;
  double* hs = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  if (!hs) return -1;
  for (int64_t c = 0; c < C; ++c) {
    const double ls = rg_log_sigmoid(a_param[c]);
    double d_ls = 0.0; /* dL / d log(sigmoid(a_param[c])) over every (b, t) */
    for (int64_t b = 0; b < B; ++b) {
      const int64_t row = (b * C + c) * T;
      /* hs[0] = h_{-1}, hs[t + 1] = h_t */
      hs[0] = h0 ? h0[b * C + c] : 0.0;
      for (int64_t t = 0; t < T; ++t) {
        const int64_t e = row + t;
        const double in_gate = rg_sigmoid(gate_x[e]);
        const int reset = segment_pos && segment_pos[b * T + t] == 0;
        const double log_a = reset ? 0.0 : RG_SCALE * rg_sigmoid(gate_a[e]) * ls;
        const double a = reset ? 0.0 : exp(log_a);
        const double mult = reset ? 1.0 : sqrt(-expm1(2.0 * log_a));
        hs[t + 1] = a * hs[t] + mult * (in_gate * x[e]);
      }
      double g = 0.0, a_next = 0.0;
      for (int64_t t = T - 1; t >= 0; --t) {
        const int64_t e = row + t;
        g = dh[e] + a_next * g; /* dL/dh_t */
        const double in_gate = rg_sigmoid(gate_x[e]);
        double a, d_in;
        if (segment_pos && segment_pos[b * T + t] == 0) {
          a = 0.0;
          dx[e] = g * in_gate;
          d_in = g * x[e];
          dgate_a[e] = 0.0;
        } else {
          const double r = rg_sigmoid(gate_a[e]);
          const double log_a = RG_SCALE * r * ls;
          a = exp(log_a);
          const double u = -expm1(2.0 * log_a);
          const double mult = sqrt(u);
          const double d_mult = g * in_gate * x[e];
          dx[e] = g * mult * in_gate;
          d_in = g * mult * x[e];
          const double dmult_du = 0.5 / sqrt(u > RG_U_MIN ? u : RG_U_MIN);
          const double d_a = g * hs[t] + d_mult * dmult_du * (-2.0 * a);
          const double d_log_a = d_a * a;
          dgate_a[e] = d_log_a * RG_SCALE * ls * r * (1.0 - r);
          d_ls += d_log_a * RG_SCALE * r;
        }
        dgate_x[e] = d_in * in_gate * (1.0 - in_gate);
        a_next = a;
      }
      if (dh0) dh0[b * C + c] = (T > 0 ? a_next : 0.0) * g;
    }
    /* d log(sigmoid(p)) / dp = sigmoid(-p) */
    da_param[c] = d_ls * rg_sigmoid(-a_param[c]);
  }
  free(hs);
  return 0;
}
