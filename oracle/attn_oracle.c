/*
 * attn_oracle.c - plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA path.
 *
 * What it computes is the plain definition, one attention head at a time:
 *
 *   S = tau * Q K^T                    (sj-techlog "FlashAttention 원 논문 해부",
 *                                        section "원 논문의 정의")
 *   s_ij = -inf for j > i when causal   (same page, "Q·K·V와 한 행의 의미")
 *   P = row-wise softmax(S), computed with the row maximum subtracted
 *                                       (same page, "stable softmax는 ...")
 *   O = P V,   lse_i = m_i + ln sum_j exp(s_ij - m_i)
 *                                       (wonbeomjang.kr FlashAttention-2 review,
 *                                        "개선 2: m과 l 대신 L만 저장")
 *
 * and the analytic backward of the same review, section "Backward Pass":
 *
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
 *   dS_ij = P_ij (dP_ij - D_i),  dQ = tau dS K,  dK = tau dS^T Q.
 *
 * The review writes dQ = dS K and dK = dS^T Q for S = Q K^T; with the softmax
 * scale tau inside S (first page's definition) the chain rule adds the factor
 * tau, which the finite-difference test of this oracle pins.
 *
 * There is no tiling, no online softmax and no reordering: every row's softmax
 * sees the whole row at once.  The only structure added is that work is split
 * by output row (forward, dQ) or by key column (dK, dV) so that any subset of
 * rows or columns can be evaluated on its own; the backward's column pass
 * re-evaluates P_ij = exp(s_ij - lse_i), which is the softmax definition
 * written with the row's log-normaliser.  Loops over independent rows/columns
 * carry an OpenMP pragma (ignored when compiled without -fopenmp).
 *
 * Layouts (row-major, one head):  q [nq][d], k [nk][d], v [nk][dv],
 * dO [nq][dv].  Causal masking uses top-left alignment: key j is visible to
 * query i iff j <= i.  Every row therefore sees at least key 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

static double dot(const double* a, const double* b, int64_t n) {
    double s = 0.0;
    for (int64_t t = 0; t < n; ++t) s += a[t] * b[t];
    return s;
}

/* Number of keys visible to query row i. */
static int64_t visible_keys(int64_t i, int64_t nk, int causal) {
    if (!causal) return nk;
    return (i + 1 < nk) ? i + 1 : nk;
}

/*
 * Scores, row maximum and log-normaliser for one query row.
 * s_out receives tau * q_i . k_j for the nvis visible keys.
 */
static double row_scores(const double* qi, const double* k, int64_t nvis, int64_t d,
                         double tau, double* s_out, double* m_out) {
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        s_out[j] = tau * dot(qi, k + j * d, d);
        if (s_out[j] > m) m = s_out[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < nvis; ++j) z += exp(s_out[j] - m);
    *m_out = m;
    return m + log(z);
}

/*
 * Forward for the listed query rows.
 *   rows[r] (0 <= rows[r] < nq) selects the query; o_out[r][dv], lse_out[r].
 * Returns 0, or -1 on invalid arguments / allocation failure.
 */
int oracle_attn_fwd_rows(const double* q, const double* k, const double* v,
                         int64_t nq, int64_t nk, int64_t d, int64_t dv,
                         int causal, double tau,
                         const int64_t* rows, int64_t nrows,
                         double* o_out, double* lse_out) {
    if (nq < 1 || nk < 1 || d < 1 || dv < 1 || nrows < 0) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= nq) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)nk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s) continue;
            const int64_t i = rows[r];
            const int64_t nvis = visible_keys(i, nk, causal);
            double m;
            const double lse = row_scores(q + i * d, k, nvis, d, tau, s, &m);
            double* oi = o_out + r * dv;
            for (int64_t c = 0; c < dv; ++c) oi[c] = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                const double p = exp(s[j] - lse);   /* P_ij */
                const double* vj = v + j * dv;
                for (int64_t c = 0; c < dv; ++c) oi[c] += p * vj[c];
            }
            lse_out[r] = lse;
        }
        free(s);
    }
    return failed ? -1 : 0;
}

/*
 * Backward, row pass, for the listed query rows:
 *   lse_out[r] = lse_i,   D_out[r] = sum_j P_ij dP_ij,
 *   dq_out[r][d] = tau * sum_j dS_ij k_j   (skipped when dq_out is NULL).
 */
int oracle_attn_bwd_rows(const double* q, const double* k, const double* v,
                         const double* dO,
                         int64_t nq, int64_t nk, int64_t d, int64_t dv,
                         int causal, double tau,
                         const int64_t* rows, int64_t nrows,
                         double* lse_out, double* D_out, double* dq_out) {
    if (nq < 1 || nk < 1 || d < 1 || dv < 1 || nrows < 0) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= nq) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)nk * sizeof(double));
        double* dp = (double*)malloc((size_t)nk * sizeof(double));
        if (!s || !dp) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s || !dp) continue;
            const int64_t i = rows[r];
            const int64_t nvis = visible_keys(i, nk, causal);
            double m;
            const double lse = row_scores(q + i * d, k, nvis, d, tau, s, &m);
            const double* doi = dO + i * dv;
            double D = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                s[j] = exp(s[j] - lse);                 /* s now holds P_ij */
                dp[j] = dot(doi, v + j * dv, dv);       /* dP_ij = dO_i . v_j */
                D += s[j] * dp[j];
            }
            if (dq_out) {
                double* dqi = dq_out + r * d;
                for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
                for (int64_t j = 0; j < nvis; ++j) {
                    const double ds = s[j] * (dp[j] - D);  /* dS_ij */
                    const double* kj = k + j * d;
                    for (int64_t c = 0; c < d; ++c) dqi[c] += tau * ds * kj[c];
                }
            }
            lse_out[r] = lse;
            D_out[r] = D;
        }
        free(s);
        free(dp);
    }
    return failed ? -1 : 0;
}

/*
 * Backward, column pass, for the listed key columns:
 *   dv_out[c][dv] = sum_i P_ij dO_i,   dk_out[c][d] = tau * sum_i dS_ij q_i,
 * where j = cols[c].  lse_all[nq] and D_all[nq] must hold lse_i and D_i for
 * EVERY query row (as produced by oracle_attn_bwd_rows over all rows).
 */
int oracle_attn_bwd_cols(const double* q, const double* k, const double* v,
                         const double* dO, const double* lse_all, const double* D_all,
                         int64_t nq, int64_t nk, int64_t d, int64_t dv,
                         int causal, double tau,
                         const int64_t* cols, int64_t ncols,
                         double* dk_out, double* dv_out) {
    if (nq < 1 || nk < 1 || d < 1 || dv < 1 || ncols < 0) return -1;
    for (int64_t c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= nk) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < ncols; ++c) {
        const int64_t j = cols[c];
        const double* kj = k + j * d;
        const double* vj = v + j * dv;
        double* dkj = dk_out + c * d;
        double* dvj = dv_out + c * dv;
        for (int64_t t = 0; t < d; ++t) dkj[t] = 0.0;
        for (int64_t t = 0; t < dv; ++t) dvj[t] = 0.0;
        /* Causal: key j is seen by rows i >= j only. */
        const int64_t i0 = causal ? j : 0;
        for (int64_t i = i0; i < nq; ++i) {
            const double* qi = q + i * d;
            const double* doi = dO + i * dv;
            const double p = exp(tau * dot(qi, kj, d) - lse_all[i]);   /* P_ij */
            const double dp = dot(doi, vj, dv);                         /* dP_ij */
            const double ds = p * (dp - D_all[i]);                      /* dS_ij */
            for (int64_t t = 0; t < dv; ++t) dvj[t] += p * doi[t];
            for (int64_t t = 0; t < d; ++t) dkj[t] += tau * ds * qi[t];
        }
    }
    return 0;
}

/* Threads the parallel loops above may use (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
