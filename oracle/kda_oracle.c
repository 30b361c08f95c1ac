/*
 * KDA forward oracle: plain fp64 token-by-token recurrence on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * CUDA path is checked against.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.  It
 * shares no code, header or constant with the CUDA library.
 *
 * What it computes (Kimi Delta Attention, a gated delta rule whose decay is a
 * per-key-channel diagonal).  For every sequence n and head h, with a state
 * S in R^{V x K} (row = value index, column = key index, the [N,H,V,K] state
 * layout of the "Core Kernel API flashkda.fwd" table on the FlashKDA page):
 *
 *   a_t   = gate(g_t + dt_bias[h])          (per key channel, natural log)
 *   beta  = sigmoid(beta logit)             (flashkda.fwd table, "beta")
 *   q,k   <- q/sqrt(|q|^2+eps), k/sqrt(..)  (only with in-kernel L2 norm)
 *   S'    = S * Diag(exp(a_t))              (decay the key columns)
 *   S     = S' + beta * (v_t - S' k_t) k_t^T  (delta-rule write)
 *   o_t   = scale * S q_t                   (read-out after the write)
 *
 * Gate forms (fla-kda SKILL.md, "Gate contracts"; fla-kda skill page):
 *   safe     : a = lower_bound * sigmoid(exp(A_log) * z), A_log omitted -> 1
 *   unsafe   : a = -exp(A_log) * softplus(z)
 *   logspace : a = g as given (the caller's log-space decay: chunk_kda without
 *              the in-kernel gate); dt_bias and A_log are not used
 * beta is taken as logits (beta = sigmoid(logit)) or, with beta_is_prob, as
 * beta itself (the "beta activation" mode of the same checklist).
 *
 * Everything is evaluated in double precision from the given inputs (bf16
 * inputs reach this code already widened to float, which is exact).  No
 * blocking, chunking or reordering: one token at a time, in order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_GATE_SAFE 1
#define ORACLE_GATE_UNSAFE 2
#define ORACLE_GATE_LOGSPACE 3

/* sigmoid in a form that does not overflow for large |x| */
static double oracle_sigmoid(double x) {
  if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
  double e = exp(x);
  return e / (1.0 + e);
}

/* softplus(x) = log(1 + e^x), written without overflow and without any
 * threshold shortcut */
static double oracle_softplus(double x) {
  return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/*
 * Run the recurrence for a list of (sequence, head) units.
 *
 * q,k,g : [total_tokens, H, K] float    v : [total_tokens, H, V] float
 * beta  : [total_tokens, H] float (logits, or beta itself with beta_is_prob)
 * A_log : [H] float or NULL (NULL allowed only with the safe gate; unused by logspace)
 * dt_bias : [H, K] float or NULL (NULL -> 0)
 * init  : [N, H, V, K] float or NULL (NULL -> zero state)
 * bos   : [N+1] token offsets of the sequences (bos[n]..bos[n+1])
 * out   : [total_tokens, H, V] double; only rows of the listed units are written
 * final : [N, H, V, K] double or NULL; only listed units are written
 * units : list of n*H+h, or NULL for every unit
 * Returns 0, or -1 on an argument error.
 */
int kda_oracle_fwd(const float *q, const float *k, const float *v, const float *g,
                   const float *beta, double scale, const float *A_log,
                   const float *dt_bias, double lower_bound, int gate_mode,
                   int beta_is_prob, int qk_l2norm, double l2_eps, const float *init,
                   double *out, double *final_state, const int64_t *bos, int64_t N,
                   int64_t H, int64_t K, int64_t V, const int64_t *units, int64_t n_units,
                   int n_threads) {
  if (!q || !k || !v || !g || !beta || !out || !bos) return -1;
  if (gate_mode != ORACLE_GATE_SAFE && gate_mode != ORACLE_GATE_UNSAFE &&
      gate_mode != ORACLE_GATE_LOGSPACE)
    return -1;
  if (gate_mode == ORACLE_GATE_UNSAFE && !A_log) return -1;
  if (K <= 0 || V <= 0 || H <= 0 || N < 0) return -1;
  int64_t total_units = units ? n_units : N * H;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double *S = (double *)malloc(sizeof(double) * (size_t)(V * K));
    double *qt = (double *)malloc(sizeof(double) * (size_t)K);
    double *kt = (double *)malloc(sizeof(double) * (size_t)K);
    double *dec = (double *)malloc(sizeof(double) * (size_t)K);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < total_units; ++u) {
      int64_t unit = units ? units[u] : u;
      int64_t n = unit / H, h = unit % H;
      /* initial state */
      for (int64_t i = 0; i < V * K; ++i)
        S[i] = init ? (double)init[(n * H + h) * V * K + i] : 0.0;
      double amul = A_log ? exp((double)A_log[h]) : 1.0;
      for (int64_t t = bos[n]; t < bos[n + 1]; ++t) {
        const float *qr = q + (t * H + h) * K;
        const float *kr = k + (t * H + h) * K;
        const float *vr = v + (t * H + h) * V;
        const float *gr = g + (t * H + h) * K;
        double b = beta_is_prob ? (double)beta[t * H + h] : oracle_sigmoid((double)beta[t * H + h]);
        /* gate activation, per key channel */
        for (int64_t c = 0; c < K; ++c) {
          double z = (double)gr[c] + (dt_bias ? (double)dt_bias[h * K + c] : 0.0);
          double a = (gate_mode == ORACLE_GATE_LOGSPACE) ? (double)gr[c]
                     : (gate_mode == ORACLE_GATE_SAFE) ? lower_bound * oracle_sigmoid(amul * z)
                                                       : -amul * oracle_softplus(z);
          dec[c] = exp(a);
        }
        /* optional L2 normalisation of q and k */
        double nq = 0.0, nk = 0.0;
        for (int64_t c = 0; c < K; ++c) {
          qt[c] = (double)qr[c];
          kt[c] = (double)kr[c];
          nq += qt[c] * qt[c];
          nk += kt[c] * kt[c];
        }
        if (qk_l2norm) {
          double rq = 1.0 / sqrt(nq + l2_eps), rk = 1.0 / sqrt(nk + l2_eps);
          for (int64_t c = 0; c < K; ++c) {
            qt[c] *= rq;
            kt[c] *= rk;
          }
        }
        /* decay, delta write, read-out; rows of S are independent */
        for (int64_t r = 0; r < V; ++r) {
          double *Sr = S + r * K;
          double pred = 0.0;
          for (int64_t c = 0; c < K; ++c) {
            Sr[c] *= dec[c];
            pred += Sr[c] * kt[c];
          }
          double w = b * ((double)vr[r] - pred);
          double o = 0.0;
          for (int64_t c = 0; c < K; ++c) {
            Sr[c] += w * kt[c];
            o += Sr[c] * qt[c];
          }
          out[(t * H + h) * V + r] = scale * o;
        }
      }
      if (final_state)
        memcpy(final_state + (n * H + h) * V * K, S, sizeof(double) * (size_t)(V * K));
    }
    free(S);
    free(qt);
    free(kt);
    free(dec);
  }
  return 0;
}

/* Threads the OpenMP runtime would use (for reporting). */
int kda_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
