/*
 * oal_oracle.c -- plain, slow, fp64 CPU oracle for OAL causal attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may link, load or call this file.  Only the tests,
 * the package's smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA sources.
 *
 * Source of the method: "Not All Dimensions Are Equal: Outlier-Aware
 * Attention Linearization with Grouped Quadratic Kernels" (arXiv:2610.13674),
 * cited below as [OAL] with section / equation numbers.
 *
 *   x_r   = q_r k_r / sqrt(d_h)                      [OAL] Sec. 4.1
 *   s_g   = sum_{r in group g} x_r,  s_bar = [1, s_1..s_G]   [OAL] Sec. 4.2
 *   kappa = eps + s_bar^T L L^T s_bar               [OAL] Sec. 4.3, Eq. (7)
 *   y_i   = sum_{j<=i} kappa(q_i,k_j) v_j / sum_{j<=i} kappa(q_i,k_j)
 *                                                   [OAL] Sec. 2, Eq. (1);
 *                                                   App. D, Eq. (25)
 *
 * Three independent evaluations live here:
 *   oal_oracle_direct     -- the plain definition, pair by pair (Eq. 7 and
 *                            the normalised causal sum).  O(T^2 d) per head.
 *   oal_oracle_recurrent  -- Algorithm 1's causal-evaluation stage: the
 *                            H0/H1/H2 prefix states of Eq. (5) and the
 *                            readout of Eq. (6), token by token, in fp64,
 *                            with the coefficient map of Sec. 4.3.
 *   oal_oracle_expand_coeffs -- the coefficient map of Sec. 4.3 rounded to
 *                            fp32 under a fixed rule (the pages give none;
 *                            the rule is stated at the function).
 *
 * Conventions fixed where the pages leave them open:
 *   - causality is inclusive (j <= i), Eq. (5) and Algorithm 1 update the
 *     states before the readout of the same token;
 *   - grouped-query attention maps query head h to key/value head
 *     h / (Hq / Hkv) (contiguous blocks of query heads share a KV head);
 *   - group 0 is the constant entry of s_bar; groups 1..G label the d
 *     dimensions (a group may be empty, it then never contributes);
 *   - only the lower triangle of L is read (L is lower-triangular).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (see build.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* L is [Hq][G+1][G+1] row-major; read only entries with column <= row. */
static double l_at(const double *Lh, int G, int row, int col) {
  return (col <= row) ? Lh[(size_t)row * (G + 1) + col] : 0.0;
}

static int check_shapes(int B, int Hq, int Hkv, int T, int d, int dv, int G) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || dv <= 0 || G <= 0)
    return ORACLE_BAD_ARG;
  if (Hq % Hkv != 0) return ORACLE_BAD_ARG;
  return ORACLE_OK;
}

static int check_groups(const int32_t *group, int Hq, int d, int G) {
  for (size_t n = 0; n < (size_t)Hq * d; ++n)
    if (group[n] < 1 || group[n] > G) return ORACLE_BAD_ARG;
  return ORACLE_OK;
}

/*
 * kappa(q, k) = eps + || L^T s_bar ||^2  ([OAL] Eq. (7): s_bar^T L L^T s_bar
 * is the squared norm of L^T s_bar).  s_bar is built from the group sums of
 * x_r = q_r k_r / sqrt(d) (Sec. 4.1-4.2).  `sbar` and `w` are scratch of
 * length G+1.
 */
static double kappa_pair(const double *q, const double *k, int d,
                         const int32_t *grp, const double *Lh, int G,
                         double eps, double *sbar, double *w) {
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  sbar[0] = 1.0;
  for (int g = 1; g <= G; ++g) sbar[g] = 0.0;
  for (int r = 0; r < d; ++r) sbar[grp[r]] += q[r] * k[r] * inv_sqrt_d;
  double quad = 0.0;
  for (int c = 0; c <= G; ++c) {
    double wc = 0.0; /* (L^T s_bar)_c = sum_g L[g][c] s_bar[g] */
    for (int g = c; g <= G; ++g) wc += l_at(Lh, G, g, c) * sbar[g];
    w[c] = wc;
    quad += wc * wc;
  }
  return eps + quad;
}

/*
 * Direct evaluation of the normalised causal kernel average.
 *
 * Q [B][Hq][T][d], K [B][Hkv][T][d], V [B][Hkv][T][dv], all fp64.
 * L [Hq][G+1][G+1] fp64, group [Hq][d] int32 with values 1..G.
 * rows: optional list of flat row ids (b*Hq + h)*T + i; if NULL every row is
 * evaluated and Y is [B][Hq][T][dv]; otherwise Y is [nrows][dv].
 * min_kappa (optional): smallest kappa met over all evaluated pairs.
 * nthreads <= 0 uses the OpenMP default.
 */
int oal_oracle_direct(const double *Q, const double *K, const double *V,
                      int B, int Hq, int Hkv, int T, int d, int dv,
                      const double *L, const int32_t *group, int G, double eps,
                      const int64_t *rows, int64_t nrows, double *Y,
                      double *min_kappa, int nthreads) {
  if (check_shapes(B, Hq, Hkv, T, d, dv, G) != ORACLE_OK) return ORACLE_BAD_ARG;
  if (check_groups(group, Hq, d, G) != ORACLE_OK) return ORACLE_BAD_ARG;
  const int64_t total = (int64_t)B * Hq * T;
  const int64_t n = rows ? nrows : total;
  const int rho = Hq / Hkv;
  double global_min = INFINITY;
  int status = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double *sbar = (double *)malloc(sizeof(double) * (G + 1));
    double *w = (double *)malloc(sizeof(double) * (G + 1));
    double *num = (double *)malloc(sizeof(double) * dv);
    double local_min = INFINITY;
    const int have_scratch = (sbar && w && num);
#pragma omp for schedule(dynamic, 16)
    for (int64_t idx = 0; idx < n; ++idx) {
      const int64_t row = rows ? rows[idx] : idx;
      double *y = Y + (size_t)idx * dv;
      if (!have_scratch || row < 0 || row >= total) {
        for (int c = 0; c < dv; ++c) y[c] = NAN;
#pragma omp atomic write
        status = have_scratch ? ORACLE_BAD_ARG : ORACLE_NO_MEMORY;
        continue;
      }
      const int i = (int)(row % T);
      const int h = (int)((row / T) % Hq);
      const int b = (int)(row / ((int64_t)T * Hq));
      const int kv = h / rho;
      const double *q = Q + (((size_t)b * Hq + h) * T + i) * d;
      const double *Kb = K + ((size_t)b * Hkv + kv) * (size_t)T * d;
      const double *Vb = V + ((size_t)b * Hkv + kv) * (size_t)T * dv;
      const double *Lh = L + (size_t)h * (G + 1) * (G + 1);
      const int32_t *grp = group + (size_t)h * d;
      double den = 0.0;
      for (int c = 0; c < dv; ++c) num[c] = 0.0;
      for (int j = 0; j <= i; ++j) { /* inclusive causal prefix */
        const double kap = kappa_pair(q, Kb + (size_t)j * d, d, grp, Lh, G,
                                      eps, sbar, w);
        if (kap < local_min) local_min = kap;
        const double *v = Vb + (size_t)j * dv;
        for (int c = 0; c < dv; ++c) num[c] += kap * v[c];
        den += kap;
      }
      for (int c = 0; c < dv; ++c) y[c] = num[c] / den;
    }
#pragma omp critical
    {
      if (local_min < global_min) global_min = local_min;
    }
    free(sbar);
    free(w);
    free(num);
  }
  if (min_kappa) *min_kappa = global_min;
  return status;
}

/*
 * Coefficient map of [OAL] Sec. 4.3 in fp64:  M = L L^T,
 *   a = eps + M_00,  b_r = 2 M_{0,g(r)},  C_rt = M_{g(r),g(t)}.
 * Fills a [1], b [d], C [d*d] for one head.
 */
static void coeffs_fp64(const double *Lh, const int32_t *grp, int G, int d,
                        double eps, double *M, double *a, double *b, double *C) {
  for (int g = 0; g <= G; ++g)
    for (int h = 0; h <= G; ++h) {
      double m = 0.0;
      for (int c = 0; c <= G; ++c) m += l_at(Lh, G, g, c) * l_at(Lh, G, h, c);
      M[g * (G + 1) + h] = m;
    }
  *a = eps + M[0];
  for (int r = 0; r < d; ++r) b[r] = 2.0 * M[grp[r]];
  for (int r = 0; r < d; ++r)
    for (int t = 0; t < d; ++t)
      C[(size_t)r * d + t] = M[grp[r] * (G + 1) + grp[t]];
}

/* Ordered-pair state layout (rows of length dv+1):
 *   row 0            H0
 *   row 1 + r        H1_r
 *   row 1 + d + r*d + t  H2_rt                  ([OAL] Eq. (5))        */
static size_t full_rows(int d) { return 1 + (size_t)d + (size_t)d * d; }

/*
 * [OAL] Algorithm 1, causal-evaluation stage, in fp64.  For each (b, kv)
 * the states are updated token by token (u = [v; 1]; H0 += u;
 * H1_r += k_r u; H2_rt += k_r k_t u) and every query head sharing that KV
 * head reads out Eq. (6):
 *   u~ = a H0 + (1/sqrt d) sum_r b_r q_r H1_r + (1/d) sum_{r,t} C_rt q_r q_t H2_rt
 *   y  = u~[0:dv] / u~[dv].
 * The coefficients are the exact fp64 map of Sec. 4.3 (not the fp32 tables).
 *
 * S0 (optional) [B][Hkv][full_rows][dv+1]: initial states (zero if NULL).
 * Y  [B][Hq][T][dv];  S_out (optional): the states after token T-1.
 */
int oal_oracle_recurrent(const double *Q, const double *K, const double *V,
                         int B, int Hq, int Hkv, int T, int d, int dv,
                         const double *L, const int32_t *group, int G,
                         double eps, const double *S0, double *Y,
                         double *S_out) {
  if (check_shapes(B, Hq, Hkv, T, d, dv, G) != ORACLE_OK) return ORACLE_BAD_ARG;
  if (check_groups(group, Hq, d, G) != ORACLE_OK) return ORACLE_BAD_ARG;
  const int rho = Hq / Hkv;
  const int U = dv + 1;
  const size_t F = full_rows(d);
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  const double inv_d = 1.0 / (double)d;
  double *S = (double *)malloc(sizeof(double) * F * U);
  double *M = (double *)malloc(sizeof(double) * (G + 1) * (G + 1));
  double *a = (double *)malloc(sizeof(double) * Hq);
  double *b = (double *)malloc(sizeof(double) * (size_t)Hq * d);
  double *C = (double *)malloc(sizeof(double) * (size_t)Hq * d * d);
  double *u = (double *)malloc(sizeof(double) * U);
  double *ut = (double *)malloc(sizeof(double) * U);
  if (!S || !M || !a || !b || !C || !u || !ut) {
    free(S); free(M); free(a); free(b); free(C); free(u); free(ut);
    return ORACLE_NO_MEMORY;
  }
  for (int h = 0; h < Hq; ++h)
    coeffs_fp64(L + (size_t)h * (G + 1) * (G + 1), group + (size_t)h * d, G, d,
                eps, M, &a[h], b + (size_t)h * d, C + (size_t)h * d * d);

  for (int bb = 0; bb < B; ++bb)
    for (int kv = 0; kv < Hkv; ++kv) {
      const size_t unit = (size_t)bb * Hkv + kv;
      if (S0) memcpy(S, S0 + unit * F * U, sizeof(double) * F * U);
      else memset(S, 0, sizeof(double) * F * U);
      for (int i = 0; i < T; ++i) {
        const double *k = K + (unit * T + i) * d;
        const double *v = V + (unit * T + i) * dv;
        for (int c = 0; c < dv; ++c) u[c] = v[c];
        u[dv] = 1.0;
        /* Algorithm 1, state updates */
        for (int c = 0; c < U; ++c) S[c] += u[c];
        for (int r = 0; r < d; ++r)
          for (int c = 0; c < U; ++c) S[(1 + r) * U + c] += k[r] * u[c];
        for (int r = 0; r < d; ++r)
          for (int t = 0; t < d; ++t) {
            double *row = S + (1 + d + (size_t)r * d + t) * U;
            const double kk = k[r] * k[t];
            for (int c = 0; c < U; ++c) row[c] += kk * u[c];
          }
        /* Algorithm 1, readout of Eq. (6) for each query head of this KV head */
        for (int h = kv * rho; h < (kv + 1) * rho; ++h) {
          const double *q = Q + (((size_t)bb * Hq + h) * T + i) * d;
          const double *bh = b + (size_t)h * d;
          const double *Ch = C + (size_t)h * d * d;
          for (int c = 0; c < U; ++c) ut[c] = a[h] * S[c];
          for (int r = 0; r < d; ++r) {
            const double wr = inv_sqrt_d * bh[r] * q[r];
            for (int c = 0; c < U; ++c) ut[c] += wr * S[(1 + r) * U + c];
          }
          for (int r = 0; r < d; ++r)
            for (int t = 0; t < d; ++t) {
              const double wrt = inv_d * Ch[(size_t)r * d + t] * q[r] * q[t];
              const double *row = S + (1 + d + (size_t)r * d + t) * U;
              for (int c = 0; c < U; ++c) ut[c] += wrt * row[c];
            }
          double *y = Y + (((size_t)bb * Hq + h) * T + i) * dv;
          for (int c = 0; c < dv; ++c) y[c] = ut[c] / ut[dv];
        }
      }
      if (S_out) memcpy(S_out + unit * F * U, S, sizeof(double) * F * U);
    }
  free(S); free(M); free(a); free(b); free(C); free(u); free(ut);
  return ORACLE_OK;
}

/*
 * fp32 coefficient tables of [OAL] Sec. 4.3, under a fixed rounding rule
 * (the pages give none):
 *   M_gh = sum_{c=0}^{min(g,h)} L[g][c] * L[h][c], in fp64, c ascending
 *          (each product of two fp32 values is exact in fp64);
 *   a    = (float)((double)eps + M_00)
 *   b_r  = (float)(2 M_{0,g(r)})
 *   C_rt = (float)M_{g(r),g(t)}                   (full layout, d*d)
 *   or, packed (r <= t, row-major upper triangle, idx = r*d - r(r-1)/2 + t-r):
 *   C'_rt = (float)((r == t ? 1 : 2) * M_{g(r),g(t)})   ([OAL] App. D,
 *          "Exact state and parameter counts": off-diagonal pairs carry
 *          multiplicity two in the packed readout)
 * all conversions round to nearest even.
 *
 * L [Hq][G+1][G+1] fp32, group [Hq][d]; a [Hq], b [Hq][d],
 * C [Hq][d*d] (packed == 0) or [Hq][d(d+1)/2] (packed == 1).
 */
int oal_oracle_expand_coeffs(const float *L, const int32_t *group, int Hq,
                             int G, int d, float eps, int packed, float *a,
                             float *b, float *C) {
  if (Hq <= 0 || G <= 0 || d <= 0) return ORACLE_BAD_ARG;
  if (check_groups(group, Hq, d, G) != ORACLE_OK) return ORACLE_BAD_ARG;
  const int G1 = G + 1;
  double *M = (double *)malloc(sizeof(double) * G1 * G1);
  if (!M) return ORACLE_NO_MEMORY;
  const size_t csize = packed ? (size_t)d * (d + 1) / 2 : (size_t)d * d;
  for (int h = 0; h < Hq; ++h) {
    const float *Lh = L + (size_t)h * G1 * G1;
    const int32_t *grp = group + (size_t)h * d;
    for (int g = 0; g < G1; ++g)
      for (int hh = 0; hh < G1; ++hh) {
        const int cmax = g < hh ? g : hh;
        double m = 0.0;
        for (int c = 0; c <= cmax; ++c)
          m = m + (double)Lh[g * G1 + c] * (double)Lh[hh * G1 + c];
        M[g * G1 + hh] = m;
      }
    a[h] = (float)((double)eps + M[0]);
    for (int r = 0; r < d; ++r) b[(size_t)h * d + r] = (float)(2.0 * M[grp[r]]);
    float *Ch = C + (size_t)h * csize;
    if (!packed) {
      for (int r = 0; r < d; ++r)
        for (int t = 0; t < d; ++t)
          Ch[(size_t)r * d + t] = (float)M[grp[r] * G1 + grp[t]];
    } else {
      size_t idx = 0;
      for (int r = 0; r < d; ++r)
        for (int t = r; t < d; ++t)
          Ch[idx++] = (float)((r == t ? 1.0 : 2.0) * M[grp[r] * G1 + grp[t]]);
    }
  }
  free(M);
  return ORACLE_OK;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oal_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
