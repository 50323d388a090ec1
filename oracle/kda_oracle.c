/*
 * CPU fp64 oracle for the chunk-parallel Kimi Delta Attention (KDA) forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the test suite, the
 * package smoke check and the benchmark's CPU-baseline leg load it.  It shares
 * no code, header, table or constant with the CUDA library, and the CUDA
 * library never calls it.
 *
 * What it computes is the token-by-token delta-rule recurrence with a
 * per-channel (diagonal) decay:
 *
 *     S_t = Diag(alpha_t) S_{t-1} - beta_t k_t (k_t^T Diag(alpha_t) S_{t-1}) + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * with S_t a K x V matrix (d_k x d_v layout, as in "KDA reading notes:
 * Implementation Notes for KDA in FLA", forward pass, step 4) and
 * alpha_t = exp(g'_t), g'_t the activated log-decay gate.  The chunk-parallel
 * form of the same notes (forward steps 1-5) is an exact reorganisation of
 * this recurrence; the oracle deliberately takes the token form, which has no
 * blocking, no triangular solve and no exponent-range tricks.
 *
 * Gate activation ("FLA-KDA engineering notes", section 2 "gate input
 * contracts"), with x = g + dt_bias (dt_bias optional, treated as 0):
 *     PLAIN   : g' = -exp(A_log) * softplus(x)
 *     SAFE    : g' = lower_bound * sigmoid(exp(A_log) * x)     (A_log optional -> factor 1)
 *     PREGATED: g' = g                                           (no activation)
 * In-kernel q/k L2 norm and beta sigmoid follow section 2.2 of the same
 * notes (use_qk_l2norm_in_kernel / use_beta_sigmoid_in_kernel).
 *
 * Parity: pinned by the CPU test suite (brute-force transition products,
 * scalar closed forms, the chunk form identity, special cases).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDAO_GATE_PREGATED 0
#define KDAO_GATE_PLAIN 1
#define KDAO_GATE_SAFE 2

static double kdao_sigmoid(double x) {
  /* split form so that exp never overflows */
  if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
  double e = exp(x);
  return e / (1.0 + e);
}

static double kdao_softplus(double x) {
  /* log(1 + e^x) = max(x,0) + log1p(e^{-|x|}), exact for every finite x */
  return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* Activated gate of one element.  a_log_present / dt_present select the optional inputs. */
double kdao_gate_value(int mode, double graw, int a_log_present, double a_log,
                       int dt_present, double dt, double lower_bound) {
  double x = graw + (dt_present ? dt : 0.0);
  if (mode == KDAO_GATE_PLAIN) return -exp(a_log) * kdao_softplus(x);
  if (mode == KDAO_GATE_SAFE) {
    double a = a_log_present ? exp(a_log) : 1.0;
    return lower_bound * kdao_sigmoid(a * x);
  }
  return graw;
}

/*
 * Activated gate for a whole [ntok, HV, K] tensor.
 * g: [ntok, HV, K]; A_log: [HV] or NULL; dt_bias: [HV*K] or NULL; out: [ntok, HV, K].
 */
void kdao_gate(int mode, int64_t ntok, int HV, int K, const double* g, const double* A_log,
               const double* dt_bias, double lower_bound, double* out) {
  for (int64_t t = 0; t < ntok; ++t)
    for (int hv = 0; hv < HV; ++hv)
      for (int kk = 0; kk < K; ++kk) {
        int64_t idx = (t * HV + hv) * (int64_t)K + kk;
        out[idx] = kdao_gate_value(mode, g[idx], A_log != NULL, A_log ? A_log[hv] : 0.0,
                                   dt_bias != NULL, dt_bias ? dt_bias[(int64_t)hv * K + kk] : 0.0,
                                   lower_bound);
      }
}

/*
 * Forward pass.
 *   q,k   [B*T, H, K]   v [B*T, HV, V]   g [B*T, HV, K]   beta [B*T, HV]
 *   A_log [HV] or NULL  dt_bias [HV*K] or NULL
 *   h0    [N, HV, K, V] or NULL (zero initial state)
 *   cu_seqlens [N+1] or NULL.  With cu_seqlens, B must be 1 and sequence n spans
 *   tokens [cu[n], cu[n+1]); without it, N = B and sequence n spans [n*T, (n+1)*T).
 *   o     [B*T, HV, V]  (rows that no sequence covers are set to 0)
 *   final_state [N, HV, K, V] or NULL
 *   nthreads <= 0: OpenMP default.
 *   h_out (nullable): the state before every chunk of chunk_size tokens of every
 *   sequence ("return_intermediate_states", reading notes section 2.2), [nct][HV][K][V]
 *   with sequence n's chunks numbered after those of sequences 0..n-1.
 * Returns 0, or -1 on inconsistent arguments.
 */
int kdao_fwd(int B, int T, int H, int HV, int K, int V,
             const double* q, const double* k, const double* v, const double* g,
             const double* beta, const double* A_log, const double* dt_bias,
             int gate_mode, double lower_bound, double scale,
             int qk_l2norm, int beta_sigmoid, double l2_eps,
             const double* h0, const int64_t* cu_seqlens, int N,
             double* o, double* final_state, int nthreads, int chunk_size, double* h_out) {
  if (h_out != NULL && chunk_size <= 0) return -1;
  if (H <= 0 || HV <= 0 || HV % H != 0 || K <= 0 || V <= 0 || B <= 0 || T < 0) return -1;
  if (cu_seqlens != NULL && B != 1) return -1;
  if (cu_seqlens == NULL && N != B) return -1;
  const int G = HV / H;
  const int64_t ntok = (int64_t)B * T;
  memset(o, 0, sizeof(double) * (size_t)(ntok * HV * V));
  const int64_t units = (int64_t)N * HV;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int bad = 0;
#pragma omp parallel
  {
    double* S = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* qh = (double*)malloc(sizeof(double) * (size_t)K);
    double* kh = (double*)malloc(sizeof(double) * (size_t)K);
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* u = (double*)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
      const int n = (int)(unit / HV);
      const int hv = (int)(unit % HV);
      const int h = hv / G; /* value head hv reads q/k head hv / G */
      int64_t bos, eos;
      if (cu_seqlens) {
        bos = cu_seqlens[n];
        eos = cu_seqlens[n + 1];
      } else {
        bos = (int64_t)n * T;
        eos = bos + T;
      }
      if (bos < 0 || eos < bos || eos > ntok) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      if (h0)
        memcpy(S, h0 + ((int64_t)n * HV + hv) * (int64_t)K * V, sizeof(double) * (size_t)K * V);
      else
        memset(S, 0, sizeof(double) * (size_t)K * V);
      int64_t cfirst = 0; /* global index of sequence n's first chunk */
      if (h_out) {
        for (int m = 0; m < n; ++m) {
          const int64_t len = cu_seqlens ? cu_seqlens[m + 1] - cu_seqlens[m] : (int64_t)T;
          cfirst += (len + chunk_size - 1) / chunk_size;
        }
      }

      for (int64_t t = bos; t < eos; ++t) {
        if (h_out && (t - bos) % chunk_size == 0)
          memcpy(h_out + ((cfirst + (t - bos) / chunk_size) * HV + hv) * (int64_t)K * V, S,
                 sizeof(double) * (size_t)K * V);
        const double* qt = q + (t * H + h) * (int64_t)K;
        const double* kt = k + (t * H + h) * (int64_t)K;
        const double* vt = v + (t * HV + hv) * (int64_t)V;
        const double* gt = g + (t * HV + hv) * (int64_t)K;
        double qn = 1.0, kn = 1.0;
        if (qk_l2norm) {
          double sq = 0.0, sk = 0.0;
          for (int i = 0; i < K; ++i) { sq += qt[i] * qt[i]; sk += kt[i] * kt[i]; }
          qn = 1.0 / sqrt(sq + l2_eps);
          kn = 1.0 / sqrt(sk + l2_eps);
        }
        for (int i = 0; i < K; ++i) { qh[i] = qt[i] * qn; kh[i] = kt[i] * kn; }
        double b = beta[t * HV + hv];
        if (beta_sigmoid) b = kdao_sigmoid(b);

        /* S <- Diag(alpha_t) S */
        for (int i = 0; i < K; ++i) {
          double gp = kdao_gate_value(gate_mode, gt[i], A_log != NULL, A_log ? A_log[hv] : 0.0,
                                      dt_bias != NULL, dt_bias ? dt_bias[(int64_t)hv * K + i] : 0.0,
                                      lower_bound);
          double a = exp(gp);
          double* row = S + (int64_t)i * V;
          for (int j = 0; j < V; ++j) row[j] *= a;
        }
        /* p = S^T k ;  u = beta (v - p) ;  S <- S + k u^T */
        for (int j = 0; j < V; ++j) p[j] = 0.0;
        for (int i = 0; i < K; ++i) {
          const double* row = S + (int64_t)i * V;
          const double ki = kh[i];
          for (int j = 0; j < V; ++j) p[j] += ki * row[j];
        }
        for (int j = 0; j < V; ++j) u[j] = b * (vt[j] - p[j]);
        for (int i = 0; i < K; ++i) {
          double* row = S + (int64_t)i * V;
          const double ki = kh[i];
          for (int j = 0; j < V; ++j) row[j] += ki * u[j];
        }
        /* o_t = scale S^T q */
        double* ot = o + (t * HV + hv) * (int64_t)V;
        for (int j = 0; j < V; ++j) p[j] = 0.0;
        for (int i = 0; i < K; ++i) {
          const double* row = S + (int64_t)i * V;
          const double qi = qh[i];
          for (int j = 0; j < V; ++j) p[j] += qi * row[j];
        }
        for (int j = 0; j < V; ++j) ot[j] = scale * p[j];
      }
      if (final_state)
        memcpy(final_state + ((int64_t)n * HV + hv) * (int64_t)K * V, S,
               sizeof(double) * (size_t)K * V);
    }
    free(S); free(qh); free(kh); free(p); free(u);
  }
  return bad ? -1 : 0;
}

/* Threads an OpenMP parallel region would use (1 without OpenMP). */
int kdao_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
