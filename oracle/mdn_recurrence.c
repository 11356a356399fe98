/*
 * Oracle (test infrastructure only): the Momentum DeltaNet two-state token
 * recurrence, in fp64, one token at a time.
 *
 * Only the tests, the graft entry's smoke check and the bench's CPU-baseline
 * leg load this file's library.  The CUDA path shares no code with it.
 *
 * Source: "MDN: Parallelizing Stepwise Momentum for Delta Linear Attention"
 * (paper-reading slides), frame "MDN adds a momentum matrix to the delta
 * update", Eqs. (3)-(5); the same equations in the Chinese reading notes,
 * section 2.2 (boxed system).  Per head, with S, M in R^{dk x dv}:
 *
 *     p_t     = alpha_t k_t                 (read address)
 *     vres_t  = v_t - S_{t-1}^T p_t         (residual, reads the old memory)
 *     M_t     = mu_t M_{t-1} - eta_t k_t vres_t^T
 *     S_t     = alpha_t S_{t-1} - beta_t M_t
 *     o_t     = S_t^T q_t                   (read from the new memory)
 *
 * Layouts (row-major, innermost last):
 *   q, k        [T_total, H, dk]   packed tokens of all sequences
 *   v, o        [T_total, H, dv]
 *   alpha, mu, eta, beta   [T_total, H]      (beta may be NULL: beta = 1)
 *   S0, M0, S_T, M_T       [n_seq, H, dk, dv]  (S0/M0 may be NULL: zero)
 *   cu_seqlens  [n_seq + 1] host int32, cu_seqlens[0] = 0,
 *               sequence s owns tokens [cu_seqlens[s], cu_seqlens[s+1]).
 *   vres_out    [T_total, H, dv] or NULL: the residual of every token (the
 *               corrected values the slides' frame "Backward computation"
 *               says the forward saves for the gradient pass)
 * Each (sequence, head) pair is an independent chain; chains run in parallel
 * under OpenMP, tokens inside a chain strictly in order.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int mdn_oracle_abi_version(void) { return 1; }

int mdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Returns 0 on success, -1 on a bad argument, -2 on allocation failure. */
int mdn_oracle_forward_vres(const double *q, const double *k, const double *v,
                            const double *alpha, const double *mu, const double *eta,
                            const double *beta, const double *S0, const double *M0,
                            double *o, double *S_T, double *M_T, double *vres_out,
                            const int32_t *cu_seqlens, int n_seq, int H, int dk,
                            int dv, int n_threads) {
    if (!q || !k || !v || !alpha || !mu || !eta || !o || !cu_seqlens)
        return -1;
    if (n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (cu_seqlens[0] != 0) return -1;
    for (int s = 0; s < n_seq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;

    const long n_chain = (long)n_seq * H;
    const size_t state = (size_t)dk * dv;
    int bad_alloc = 0;

#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad_alloc)
    for (long chain = 0; chain < n_chain; ++chain) {
        const int s = (int)(chain / H);
        const int h = (int)(chain % H);
        double *S = (double *)malloc(state * sizeof(double));
        double *M = (double *)malloc(state * sizeof(double));
        double *vres = (double *)malloc((size_t)dv * sizeof(double));
        if (!S || !M || !vres) {
            free(S); free(M); free(vres);
            bad_alloc = 1;
            continue;
        }
        const size_t st_off = (size_t)chain * state;
        if (S0) memcpy(S, S0 + st_off, state * sizeof(double));
        else memset(S, 0, state * sizeof(double));
        if (M0) memcpy(M, M0 + st_off, state * sizeof(double));
        else memset(M, 0, state * sizeof(double));

        for (int t = cu_seqlens[s]; t < cu_seqlens[s + 1]; ++t) {
            const size_t g = (size_t)t * H + h; /* gate index */
            const double *kt = k + g * dk;
            const double *qt = q + g * dk;
            const double *vt = v + g * dv;
            double *ot = o + g * dv;
            const double a = alpha[g], m = mu[g], e = eta[g];
            const double b = beta ? beta[g] : 1.0;

            /* residual: vres = v - S^T (a k) */
            for (int j = 0; j < dv; ++j) vres[j] = vt[j];
            for (int i = 0; i < dk; ++i) {
                const double p = a * kt[i];
                const double *Srow = S + (size_t)i * dv;
                for (int j = 0; j < dv; ++j) vres[j] -= Srow[j] * p;
            }
            if (vres_out) memcpy(vres_out + g * dv, vres, (size_t)dv * sizeof(double));
            /* momentum: M = mu M - eta k vres^T */
            for (int i = 0; i < dk; ++i) {
                double *Mrow = M + (size_t)i * dv;
                const double ek = e * kt[i];
                for (int j = 0; j < dv; ++j) Mrow[j] = m * Mrow[j] - ek * vres[j];
            }
            /* memory: S = alpha S - beta M (the new M) */
            for (int i = 0; i < dk; ++i) {
                double *Srow = S + (size_t)i * dv;
                const double *Mrow = M + (size_t)i * dv;
                for (int j = 0; j < dv; ++j) Srow[j] = a * Srow[j] - b * Mrow[j];
            }
            /* output: o = S^T q (the new S) */
            for (int j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int i = 0; i < dk; ++i) {
                const double *Srow = S + (size_t)i * dv;
                for (int j = 0; j < dv; ++j) ot[j] += Srow[j] * qt[i];
            }
        }
        if (S_T) memcpy(S_T + st_off, S, state * sizeof(double));
        if (M_T) memcpy(M_T + st_off, M, state * sizeof(double));
        free(S); free(M); free(vres);
    }
    return bad_alloc ? -2 : 0;
}

int mdn_oracle_forward(const double *q, const double *k, const double *v,
                       const double *alpha, const double *mu, const double *eta,
                       const double *beta, const double *S0, const double *M0,
                       double *o, double *S_T, double *M_T,
                       const int32_t *cu_seqlens, int n_seq, int H, int dk,
                       int dv, int n_threads) {
    return mdn_oracle_forward_vres(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T,
                                   NULL, cu_seqlens, n_seq, H, dk, dv, n_threads);
}
