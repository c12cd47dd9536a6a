/*
 * Oracle for the gated temporal scan layer: plain fp64 CPU loops.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header, table or helper with the
 * CUDA library; both sides only see the same seeded inputs.
 *
 * What it computes, per sample b (notation of the pages: SH2 = trunk width,
 * D = STATE_D, K = history length, t = 0 is the oldest step and is scanned
 * first):
 *
 *   A[t,s]  = sum_j h_history[b,t,j] * W_A[j,s]        ("Custom Kernel
 *   Bv[t,s] = sum_j h_history[b,t,j] * W_B[j,s]         Optimization --
 *   C[s]    = sum_j h_s2[b,j]        * W_C[j,s]         cuBLAS Projections +
 *                                                       Batch-Parallel Scans",
 *                                                       Design 1, Step 1)
 *   x_{-1} = 0;  x_t = sigmoid(A[t]) * x_{t-1} + Bv[t]  (same section, Step 2;
 *                                                       "Custom Kernel
 *                                                       Optimization
 *                                                       Implementation Plan",
 *                                                       Task 1 Step 3)
 *   ctx[s] = C[s] * x_{K-1}[s]                          (design spec, Design 1
 *                                                       Step 2: one context
 *                                                       value per state)
 *   h_enriched[b,j] = h_s2[b,j] + tw * sum_s ctx[s] * W_O[s,j]
 *       The pages leave this output step open (design spec, Design 1 Step 3);
 *       the layer fixes it as a residual plus a [D, SH2] output projection
 *       scaled by the scalar tw.
 *
 * Backward, with g = dL/dh_enriched[b,:] (derived by the chain rule from the
 * forward above; the implementation plan's Task 2 gives the reverse scan
 * d_gate = dx * x_{t-1} * sigmoid' and dx <- dx * gate):
 *
 *   d_ctx[s]  = tw * sum_j g[j] * W_O[s,j]
 *   dW_O[s,j] += tw * ctx[s] * g[j]
 *   dC[s]     = d_ctx[s] * x_{K-1}[s]
 *   dx        = d_ctx[s] * C[s]                       (gradient wrt x_{K-1})
 *   for t = K-1 .. 0:
 *       dBv[t,s] = dx
 *       dA[t,s]  = dx * x_{t-1}[s] * sig_t * (1 - sig_t)     (x_{-1} = 0)
 *       dx       = dx * sig_t
 *   dW_A[j,s] += sum_t h_history[b,t,j] * dA[t,s]     (plan, Task 2 Step 3)
 *   dW_B[j,s] += sum_t h_history[b,t,j] * dBv[t,s]
 *   dW_C[j,s] += h_s2[b,j] * dC[s]
 *   d_h_history[b,t,j] = sum_s dA[t,s] * W_A[j,s] + dBv[t,s] * W_B[j,s]
 *   d_h_s2[b,j]        = g[j] + sum_s dC[s] * W_C[j,s]
 *
 * Weight gradients are summed per fixed block of samples and the blocks are
 * then added in block order, so the result does not depend on the number of
 * threads that ran it.
 *
 * Error scale of the weight gradients (test infrastructure, not part of the
 * layer): each weight gradient is a sum of per-sample terms (h * dA, h * dBv,
 * hs * dC, tw * ctx * g). When `abs_terms` is not NULL the backward also
 * returns, per element, the sum of the absolute values of those same terms,
 *   |dW_A|[j,s] = sum over b, t of |h[b,t,j] * dA[t,s]|   (likewise |dW_B|)
 *   |dW_C|[j,s] = sum over b of |hs[b,j] * dC[s]|
 *   |dW_O|[s,j] = sum over b of |tw * ctx[s] * g[j]|
 * (blend form: sum over b of |g[j] * context / D|). The rounding error of any
 * fp32 evaluation of a sum is bounded by a multiple of this quantity (the
 * standard bound for floating-point summation), not by the sum itself.
 * `abs_dh`, `abs_dhs2` (backward) and `abs_out` (forward) do the same for the
 * per-sample outputs: sum over s of |dA*W_A| + |dBv*W_B|, |g| + sum over s of
 * |dC*W_C| and |hs| + |tw| * sum over s of |ctx*W_O| (blend: |hs| +
 * |w| * sum over s of |ctx| / D). NULL skips any of them.
 *
 * Layouts (row-major, contiguous): h_history [B,K,SH2], h_s2 [B,SH2],
 * W_A, W_B, W_C [SH2,D], W_O [D,SH2], d_h_enriched and h_enriched [B,SH2].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define M2O_BLOCKS 64 /* fixed number of sample blocks for the dW sums */

static double sigmoid(double a) { return 1.0 / (1.0 + exp(-a)); }

/* Projections and forward scan of one sample. A, Bv, sig, x are [K,D]; C and
 * ctx are [D]. x[t] is the state after step t; sig[t] = sigmoid(A[t]) before
 * the gate scale gs (the pages' optional gate multiplier, "Custom Kernel
 * Optimization Implementation Plan", Task 1: gate *= isv_signals[11]; 1 when
 * absent), so the gate of step t is gs * sig[t]. */
static void sample_forward(const double* h, const double* hs, const double* W_A,
                           const double* W_B, const double* W_C, int K, int SH2,
                           int D, double gs, double* A, double* Bv, double* sig, double* x,
                           double* C, double* ctx) {
  for (int t = 0; t < K; t++) {
    for (int s = 0; s < D; s++) {
      double a = 0.0, bb = 0.0;
      for (int j = 0; j < SH2; j++) {
        a += h[(int64_t)t * SH2 + j] * W_A[(int64_t)j * D + s];
        bb += h[(int64_t)t * SH2 + j] * W_B[(int64_t)j * D + s];
      }
      A[t * D + s] = a;
      Bv[t * D + s] = bb;
    }
  }
  for (int s = 0; s < D; s++) {
    double c = 0.0;
    for (int j = 0; j < SH2; j++) c += hs[j] * W_C[(int64_t)j * D + s];
    C[s] = c;
  }
  for (int s = 0; s < D; s++) {
    double xs = 0.0; /* x_{-1} = 0 */
    for (int t = 0; t < K; t++) {
      double g = sigmoid(A[t * D + s]);
      sig[t * D + s] = g;
      xs = gs * g * xs + Bv[t * D + s];
      x[t * D + s] = xs;
    }
    ctx[s] = C[s] * xs;
  }
}

/* Intermediates for every sample, for tests that pin the scan itself.
 * A, Bv, x: [B,K,D]; C, ctx: [B,D]. */
int m2o_scan_state(const double* h_history, const double* h_s2, const double* W_A,
                   const double* W_B, const double* W_C, int64_t B, int K, int SH2,
                   int D, double gs, double* A, double* Bv, double* x, double* C, double* ctx) {
  if (B < 0 || K < 1 || SH2 < 1 || D < 1) return 1;
  double* sig = (double*)malloc(sizeof(double) * (size_t)K * D);
  if (!sig) return 2;
  for (int64_t b = 0; b < B; b++) {
    sample_forward(h_history + b * K * SH2, h_s2 + b * SH2, W_A, W_B, W_C, K, SH2, D, gs,
                   A + b * K * D, Bv + b * K * D, sig, x + b * K * D, C + b * D,
                   ctx + b * D);
  }
  free(sig);
  return 0;
}

/* Output step, two forms. blend == 0 (the layer's):
 *   h_enriched[j] = h_s2[j] + tw * sum_s ctx[s] * W_O[s, j].
 * blend == 1 (the pages' own, "Custom Kernel Optimization Implementation
 * Plan", Task 1 Step 3): one scalar context per sample, sum_s ctx[s], blended
 * into every feature with a per-feature weight and a 1/D scale,
 *   h_enriched[j] = h_s2[j] + w[j] * (sum_s ctx[s]) / D,
 * W_O then holds w [SH2] (NULL: every weight 1) and tw is not used. */
int m2o_forward(const double* h_history, const double* h_s2, const double* W_A,
                const double* W_B, const double* W_C, const double* W_O, double tw,
                int64_t B, int K, int SH2, int D, double gs, int blend, double* h_enriched,
                double* abs_out, int n_threads) {
  if (B < 0 || K < 1 || SH2 < 1 || D < 1) return 1;
  if (n_threads < 1) n_threads = 1;
  int fail = 0;
#pragma omp parallel num_threads(n_threads)
  {
    double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * K * D + 2 * D));
    if (!buf) {
#pragma omp atomic write
      fail = 2;
    }
#pragma omp for schedule(static)
    for (int64_t b = 0; b < B; b++) {
      if (!buf) continue;
      double *A = buf, *Bv = A + K * D, *sig = Bv + K * D, *x = sig + K * D;
      double *C = x + K * D, *ctx = C + D;
      const double* hs = h_s2 + b * SH2;
      sample_forward(h_history + b * K * SH2, hs, W_A, W_B, W_C, K, SH2, D, gs, A, Bv,
                     sig, x, C, ctx);
      if (blend) {
        double context = 0.0;
        for (int s = 0; s < D; s++) context += ctx[s];
        double acontext = 0.0;
        for (int s = 0; s < D; s++) acontext += fabs(ctx[s]);
        for (int j = 0; j < SH2; j++) {
          const double w = W_O ? W_O[j] : 1.0;
          h_enriched[b * SH2 + j] = hs[j] + w * context / D;
          if (abs_out) abs_out[b * SH2 + j] = fabs(hs[j]) + fabs(w) * acontext / D;
        }
        continue;
      }
      for (int j = 0; j < SH2; j++) {
        double o = 0.0, ao = 0.0;
        for (int s = 0; s < D; s++) {
          o += ctx[s] * W_O[(int64_t)s * SH2 + j];
          ao += fabs(ctx[s] * W_O[(int64_t)s * SH2 + j]);
        }
        h_enriched[b * SH2 + j] = hs[j] + tw * o;
        if (abs_out) abs_out[b * SH2 + j] = fabs(hs[j]) + fabs(tw) * ao;
      }
    }
    free(buf);
  }
  return fail;
}

int m2o_backward(const double* h_history, const double* h_s2, const double* W_A,
                 const double* W_B, const double* W_C, const double* W_O, double tw,
                 const double* d_h_enriched, int64_t B, int K, int SH2, int D, double gs,
                 int blend, double* d_h_history, double* d_h_s2, double* dW_A, double* dW_B,
                 double* dW_C, double* dW_O, double* abs_terms, double* abs_dh,
                 double* abs_dhs2, int n_threads) {
  if (B < 0 || K < 1 || SH2 < 1 || D < 1) return 1;
  if (n_threads < 1) n_threads = 1;
  const int64_t nw = (int64_t)SH2 * D; /* elements of each weight gradient */
  /* per-block partial sums: [block][8][nw], order dW_A, dW_B, dW_C, dW_O, then
   * the absolute-term sums of the same four */
  double* part = (double*)calloc((size_t)M2O_BLOCKS * 8 * nw, sizeof(double));
  if (!part) return 2;
  int fail = 0;
#pragma omp parallel num_threads(n_threads)
  {
    double* buf = (double*)malloc(sizeof(double) * (size_t)(6 * K * D + 5 * D));
    if (!buf) {
#pragma omp atomic write
      fail = 2;
    }
#pragma omp for schedule(dynamic, 1)
    for (int blk = 0; blk < M2O_BLOCKS; blk++) {
      if (!buf) continue;
      double* pA = part + (int64_t)blk * 8 * nw;
      double* pB = pA + nw;
      double* pC = pB + nw;
      double* pO = pC + nw; /* stored [D,SH2] like W_O */
      double* qA = pO + nw; /* absolute-term sums, same layouts */
      double* qB = qA + nw;
      double* qC = qB + nw;
      double* qO = qC + nw;
      int64_t b0 = B * blk / M2O_BLOCKS, b1 = B * (blk + 1) / M2O_BLOCKS;
      double *A = buf, *Bv = A + K * D, *sig = Bv + K * D, *x = sig + K * D;
      double *dA = x + K * D, *dBv = dA + K * D;
      double *C = dBv + K * D, *ctx = C + D, *dctx = ctx + D, *dC = dctx + D;
      for (int64_t b = b0; b < b1; b++) {
        const double* h = h_history + b * K * SH2;
        const double* hs = h_s2 + b * SH2;
        const double* g = d_h_enriched + b * SH2;
        sample_forward(h, hs, W_A, W_B, W_C, K, SH2, D, gs, A, Bv, sig, x, C, ctx);
        /* output step (blend: the scalar context's gradient is shared by every
         * state, and dW_O holds the per-feature weights' gradient, dw [SH2]) */
        if (blend) {
          double context = 0.0, dcontext = 0.0;
          for (int s = 0; s < D; s++) context += ctx[s];
          for (int j = 0; j < SH2; j++) {
            const double w = W_O ? W_O[j] : 1.0;
            dcontext += g[j] * w / D;
            pO[j] += g[j] * context / D;
            qO[j] += fabs(g[j] * context / D);
          }
          for (int s = 0; s < D; s++) {
            dctx[s] = dcontext;
            dC[s] = dcontext * x[(K - 1) * D + s];
          }
        }
        for (int s = 0; s < D && !blend; s++) {
          double acc = 0.0;
          for (int j = 0; j < SH2; j++) acc += g[j] * W_O[(int64_t)s * SH2 + j];
          dctx[s] = tw * acc;
          for (int j = 0; j < SH2; j++) {
            pO[(int64_t)s * SH2 + j] += tw * ctx[s] * g[j];
            qO[(int64_t)s * SH2 + j] += fabs(tw * ctx[s] * g[j]);
          }
          dC[s] = dctx[s] * x[(K - 1) * D + s];
        }
        /* reverse scan; the gate of step t is gs * sigmoid(A[t]) (same plan,
         * Task 2: d_gate and d_x both carry the stability factor) */
        for (int s = 0; s < D; s++) {
          double dx = dctx[s] * C[s];
          for (int t = K - 1; t >= 0; t--) {
            double gt = sig[t * D + s];
            double xprev = (t > 0) ? x[(t - 1) * D + s] : 0.0;
            dBv[t * D + s] = dx;
            dA[t * D + s] = dx * xprev * gs * gt * (1.0 - gt);
            dx = dx * gs * gt;
          }
        }
        /* weight gradients */
        for (int j = 0; j < SH2; j++) {
          for (int s = 0; s < D; s++) {
            double sa = 0.0, sb = 0.0, ua = 0.0, ub = 0.0;
            for (int t = 0; t < K; t++) {
              sa += h[(int64_t)t * SH2 + j] * dA[t * D + s];
              sb += h[(int64_t)t * SH2 + j] * dBv[t * D + s];
              ua += fabs(h[(int64_t)t * SH2 + j] * dA[t * D + s]);
              ub += fabs(h[(int64_t)t * SH2 + j] * dBv[t * D + s]);
            }
            pA[(int64_t)j * D + s] += sa;
            pB[(int64_t)j * D + s] += sb;
            pC[(int64_t)j * D + s] += hs[j] * dC[s];
            qA[(int64_t)j * D + s] += ua;
            qB[(int64_t)j * D + s] += ub;
            qC[(int64_t)j * D + s] += fabs(hs[j] * dC[s]);
          }
        }
        /* input gradients */
        for (int t = 0; t < K; t++) {
          for (int j = 0; j < SH2; j++) {
            double acc = 0.0, aacc = 0.0;
            for (int s = 0; s < D; s++) {
              acc += dA[t * D + s] * W_A[(int64_t)j * D + s] +
                     dBv[t * D + s] * W_B[(int64_t)j * D + s];
              aacc += fabs(dA[t * D + s] * W_A[(int64_t)j * D + s]) +
                      fabs(dBv[t * D + s] * W_B[(int64_t)j * D + s]);
            }
            d_h_history[(b * K + t) * SH2 + j] = acc;
            if (abs_dh) abs_dh[(b * K + t) * SH2 + j] = aacc;
          }
        }
        for (int j = 0; j < SH2; j++) {
          double acc = g[j], aacc = fabs(g[j]);
          for (int s = 0; s < D; s++) {
            acc += dC[s] * W_C[(int64_t)j * D + s];
            aacc += fabs(dC[s] * W_C[(int64_t)j * D + s]);
          }
          d_h_s2[b * SH2 + j] = acc;
          if (abs_dhs2) abs_dhs2[b * SH2 + j] = aacc;
        }
      }
    }
    free(buf);
  }
  /* combine the blocks in block order */
  for (int64_t e = 0; e < nw; e++) {
    double sa = 0.0, sb = 0.0, sc = 0.0, so = 0.0;
    double ua = 0.0, ub = 0.0, uc = 0.0, uo = 0.0;
    for (int blk = 0; blk < M2O_BLOCKS; blk++) {
      const double* p = part + (int64_t)blk * 8 * nw;
      sa += p[e];
      sb += p[nw + e];
      sc += p[2 * nw + e];
      so += p[3 * nw + e];
      ua += p[4 * nw + e];
      ub += p[5 * nw + e];
      uc += p[6 * nw + e];
      uo += p[7 * nw + e];
    }
    dW_A[e] = sa;
    dW_B[e] = sb;
    dW_C[e] = sc;
    if (!blend || e < SH2) dW_O[e] = so;
    if (abs_terms) {
      abs_terms[e] = ua;
      abs_terms[nw + e] = ub;
      abs_terms[2 * nw + e] = uc;
      if (!blend || e < SH2) abs_terms[3 * nw + e] = uo;
    }
  }
  free(part);
  return fail;
}

/*
 * Bias gradient of a fully connected layer: column sums of a row-major
 * [N, C] matrix of upstream gradients,
 *
 *   db[c] = sum over rows r = 0 .. N-1 of dy[r, c]
 *
 * ("Phase 3 Kernel Optimization Implementation Plan", Task 2: the reduction
 * over the batch of every output feature's gradient). The pages keep two
 * conventions: the main network's backward adds the sum into db, the
 * curiosity trainer (Task 3) overwrites grad_b; `accumulate` selects the
 * first (db_out = db_in + sum), else db_out = sum. One fp64 accumulator per
 * column, rows added in order.
 */
int m2o_bias_grad(const double* dy, int64_t N, int C, const double* db_in, int accumulate,
                  double* db_out) {
  if (N < 0 || C < 1 || (N > 0 && !dy) || !db_out || (accumulate && !db_in)) return 1;
  for (int c = 0; c < C; c++) {
    double acc = 0.0;
    for (int64_t r = 0; r < N; r++) acc += dy[r * C + c];
    db_out[c] = accumulate ? db_in[c] + acc : acc;
  }
  return 0;
}
