/*
 * KDA token-by-token reference recurrence, fp64.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the oracle that the CUDA path is checked against.  Only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark may build,
 * load or call it; the library's own code never does.  It shares no code,
 * header or table with the CUDA kernels.
 *
 * What it computes (per sequence n, value head h, token t; K = V = 128):
 *   gate   g~_t = lower_bound * sigmoid(exp(A_log[h]) * (g_t + dt_bias[h]))
 *          (page "mate/kda.py", chunk_kda docstring: A_log per head, dt_bias
 *          per head and channel, lower bound applied when both are given;
 *          page "verify" KdaTcVerify.kernel, step 2 "Activations": the
 *          per-channel gate is lower_bound * sigmoid(a * (g + bias)) with
 *          a = exp(a_log)).  Without A_log/dt_bias the gate input g is the
 *          log decay itself and lower_bound is not used.
 *   beta_t = sigmoid(b_t)                       ("Beta logits", chunk_kda docs)
 *   k^_t   = k_t / sqrt(|k_t|^2 + 1e-6)
 *   q~_t   = scale * q_t / sqrt(|q_t|^2 + 1e-6)  (verify page, "Probes":
 *          rsqrt(sum + 1e-6), scale applied after the norm)
 *   S     <- diag(exp(g~_t)) S                  (decay of the K rows)
 *   U_t    = beta_t (v_t - S^T k^_t)            (delta-rule correction)
 *   S     <- S + k^_t U_t^T
 *   o_t    = S^T q~_t
 * S is K x V and stored V-first ([V][K], K contiguous), as the decode page's
 * default ``state_v_first`` layout and the verify page's [slots, H, V, K]
 * state.  The value head h reads query/key head h / (Hv / Hqk).
 *
 * Parallelism: OpenMP over (sequence, head, block of 16 value columns); the
 * value columns of S evolve independently in the recurrence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KD 128
#define VB 16 /* value columns per task */

static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

int kda_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Inputs are fp32 arrays holding the (bf16-representable) input values, in
 * the flattened token-major layout:
 *   q, k [T_tot][Hqk][128], v, g [T_tot][Hv][128], b [T_tot][Hv].
 *   A_log [Hv] and dt_bias [Hv][128] (both NULL: gate input used directly).
 *   cu_seqlens [n_seqs + 1] token offsets.
 *   h0   [n_seqs][Hv][V][K] fp64 initial states, or NULL for zero.
 * Outputs (fp64, any may be NULL):
 *   out  [T_tot][Hv][V]   per-token outputs o_t
 *   hT   [n_seqs][Hv][V][K] final states
 *   corr [T_tot][Hv][V]   the correction vectors U_t
 * Returns 0, or -1 on a bad argument.
 */
int kda_oracle_recurrence(const float* q, const float* k, const float* v,
                          const float* g, const float* b, const float* A_log,
                          const float* dt_bias, const int64_t* cu_seqlens,
                          int n_seqs, int Hqk, int Hv, double scale,
                          double lower_bound, int use_qk_l2norm,
                          const double* h0, double* out, double* hT,
                          double* corr, int n_threads) {
  if (Hqk <= 0 || Hv <= 0 || Hv % Hqk != 0 || n_seqs < 0) return -1;
  if ((A_log == NULL) != (dt_bias == NULL)) return -1;
  const int ratio = Hv / Hqk;
  const int nvb = KD / VB;
  const long n_tasks = (long)n_seqs * Hv * nvb;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
  for (long task = 0; task < n_tasks; ++task) {
    const int vb = (int)(task % nvb);
    const int h = (int)((task / nvb) % Hv);
    const int n = (int)(task / ((long)nvb * Hv));
    const int hq = h / ratio;
    const int v0 = vb * VB;
    double S[VB][KD]; /* S^T rows v0..v0+VB-1 (V-first) */
    double kh[KD], qh[KD], decay[KD];

    for (int j = 0; j < VB; ++j)
      for (int c = 0; c < KD; ++c)
        S[j][c] = h0 ? h0[(((long)n * Hv + h) * KD + v0 + j) * KD + c] : 0.0;

    const double a_h = A_log ? exp((double)A_log[h]) : 0.0;
    for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
      const float* qt = q + (t * Hqk + hq) * KD;
      const float* kt = k + (t * Hqk + hq) * KD;
      const float* vt = v + (t * Hv + h) * KD;
      const float* gt = g + (t * Hv + h) * KD;
      const double beta = sigmoid_d((double)b[t * Hv + h]);

      /* gate (log decay per key channel) */
      for (int c = 0; c < KD; ++c) {
        double gate;
        if (A_log)
          gate = lower_bound *
                 sigmoid_d(a_h * ((double)gt[c] + (double)dt_bias[h * KD + c]));
        else
          gate = (double)gt[c];
        decay[c] = exp(gate);
      }
      /* L2 norms */
      double sq = 0.0, sk = 0.0;
      for (int c = 0; c < KD; ++c) {
        sq += (double)qt[c] * (double)qt[c];
        sk += (double)kt[c] * (double)kt[c];
      }
      const double rq = use_qk_l2norm ? 1.0 / sqrt(sq + 1e-6) : 1.0;
      const double rk = use_qk_l2norm ? 1.0 / sqrt(sk + 1e-6) : 1.0;
      for (int c = 0; c < KD; ++c) {
        kh[c] = (double)kt[c] * rk;
        qh[c] = scale * (double)qt[c] * rq;
      }
      for (int j = 0; j < VB; ++j) {
        double* s = S[j];
        /* S <- diag(exp(gate)) S : row j of S^T scales channel c */
        for (int c = 0; c < KD; ++c) s[c] *= decay[c];
        /* U = beta (v - S^T k^) */
        double sk_dot = 0.0;
        for (int c = 0; c < KD; ++c) sk_dot += s[c] * kh[c];
        const double u = beta * ((double)vt[v0 + j] - sk_dot);
        /* S <- S + k^ U^T */
        for (int c = 0; c < KD; ++c) s[c] += kh[c] * u;
        /* o = S^T q~ */
        double o = 0.0;
        for (int c = 0; c < KD; ++c) o += s[c] * qh[c];
        if (out) out[(t * Hv + h) * KD + v0 + j] = o;
        if (corr) corr[(t * Hv + h) * KD + v0 + j] = u;
      }
    }
    if (hT)
      for (int j = 0; j < VB; ++j)
        for (int c = 0; c < KD; ++c)
          hT[(((long)n * Hv + h) * KD + v0 + j) * KD + c] = S[j][c];
  }
  return 0;
}
