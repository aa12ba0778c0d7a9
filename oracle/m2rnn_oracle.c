/*
 * m2rnn_oracle.c -- plain fp64 CPU oracle for the M2RNN recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Source of the arithmetic: "M2RNN: Non-Linear RNNs with Matrix-Valued States
 * for Scalable Language Modeling" (arXiv 2603.14360v2), as discussed in the
 * slide deck "M2RNN research paper discussion":
 *   - frame "Write, transform, retain, and read a matrix state", paper
 *     Eqs. (10)-(12):
 *         Z_t = tanh(H_{t-1} W + k_t v_t^T)
 *         H_t = f_t H_{t-1} + (1 - f_t) Z_t
 *         y_t = H_t^T q_t + w_r (.) v_t
 *     with H_t, Z_t in R^{K x V}, W in R^{V x V}, H_0 = 0 (or a given H0).
 *   - frame "Shared queries and keys buy more recurrent capacity": q, k are
 *     shared by the N value heads (N_q = N_k = 1); v, f, W, w_r are per head.
 *   - backup frame "Backup: the recurrent gradient needs both paths": with
 *     u_t = dL/dy_t and C_t the gradient arriving from later steps,
 *         R_t     = C_t + q_t u_t^T
 *         D_t     = ((1 - f_t) R_t) (.) (1 - Z_t (.) Z_t)
 *         C_{t-1} = f_t R_t + D_t W^T
 *         dL/df_t = <R_t, H_{t-1} - Z_t>_F
 *         dL/dW   = sum_t H_{t-1}^T D_t
 *     The same frame notes that the value residual contributes further
 *     gradients; those (dq, dk, dv, dw_r) follow from Eqs. (10)-(12) by the
 *     chain rule:
 *         dk_t  = sum_n D_t v_t          (k enters only through k_t v_t^T)
 *         dv_t  = D_t^T k_t + w_r (.) u_t
 *         dq_t  = sum_n H_t u_t          (q enters only through H_t^T q_t)
 *         dw_r  = sum_{b,t} u_t (.) v_t
 *         dH_0  = C_0
 *     The printed "Algorithm 2" of the paper is not followed: the deck states
 *     it drops C_t and mis-updates the state gradient.
 *
 * Readings taken where the pages are silent:
 *   - W acts on the right of H: (H W)_{i,j} = sum_l H_{i,l} W_{l,j}; W is
 *     stored row-major as W[l][j] ("W mixes value channels within each row").
 *   - y_t reads the updated state H_t, not H_{t-1}; no query scaling.
 *   - f is given directly per (b, t, n); the gate formula is not applied here.
 *   - C_T = dH_T when given, else 0; exact gradients, no clipping.
 *
 * Layouts (row-major, contiguous):
 *   q, k [B,T,K]   v [B,T,N,V]   f [B,T,N]   W [N,V,V]   w_r [N,V]
 *   H0, HT, dHT, dH0 [B,N,K,V]   y, dy, dv [B,T,N,V]   dq, dk [B,T,K]
 *   df [B,T,N]   dW [N,V,V]   dw_r [N,V]
 *
 * Parallelism: OpenMP over independent (b, n) pairs.  Every cross-head or
 * cross-batch sum is done afterwards, serially, in a fixed order.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX2(a, b, nb) ((size_t)(a) * (size_t)(nb) + (size_t)(b))

int m2rnn_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One forward step of Eqs. (10)-(12) for one (b, n):
 *   Hprev [K,V] -> Z [K,V], Hnext [K,V]. */
static void oracle_step(int K, int V, const double *Hprev, const double *Wn,
                        const double *kt, const double *vt, double ft,
                        double *Z, double *Hnext)
{
    for (int i = 0; i < K; ++i) {
        for (int j = 0; j < V; ++j) {
            double a = 0.0;
            for (int l = 0; l < V; ++l)
                a += Hprev[IDX2(i, l, V)] * Wn[IDX2(l, j, V)];
            a += kt[i] * vt[j];
            Z[IDX2(i, j, V)] = tanh(a);
        }
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            Hnext[IDX2(i, j, V)] = ft * Hprev[IDX2(i, j, V)] + (1.0 - ft) * Z[IDX2(i, j, V)];
}

/* Forward pass.  y and HT are written; HT and H0 may be NULL.  If `states`
 * is non-NULL it receives every state H_0..H_T as [B,N,T+1,K,V]. */
int m2rnn_oracle_fwd(int B, int T, int N, int K, int V,
                     const double *q, const double *k, const double *v,
                     const double *f, const double *W, const double *w_r,
                     const double *H0, double *y, double *HT, double *states)
{
    if (B < 0 || T < 0 || N < 0 || K <= 0 || V <= 0) return -1;
    const size_t KV = (size_t)K * V;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bn = 0; bn < (long)B * N; ++bn) {
        const int b = (int)(bn / N), n = (int)(bn % N);
        double *H = (double *)malloc(KV * sizeof(double));
        double *Hn = (double *)malloc(KV * sizeof(double));
        double *Z = (double *)malloc(KV * sizeof(double));
        if (!H || !Hn || !Z) {
#pragma omp atomic write
            err = -2;
            free(H); free(Hn); free(Z);
            continue;
        }
        const double *Wn = W + (size_t)n * V * V;
        const double *wrn = w_r + (size_t)n * V;
        if (H0) memcpy(H, H0 + IDX2(b, n, N) * KV, KV * sizeof(double));
        else memset(H, 0, KV * sizeof(double));
        if (states) memcpy(states + (IDX2(b, n, N) * (size_t)(T + 1)) * KV, H, KV * sizeof(double));
        for (int t = 0; t < T; ++t) {
            const double *qt = q + IDX2(b, t, T) * K;
            const double *kt = k + IDX2(b, t, T) * K;
            const double *vt = v + (IDX2(b, t, T) * N + n) * V;
            const double ft = f[IDX2(b, t, T) * N + n];
            oracle_step(K, V, H, Wn, kt, vt, ft, Z, Hn);
            double *tmp = H; H = Hn; Hn = tmp;
            double *yt = y + (IDX2(b, t, T) * N + n) * V;
            for (int j = 0; j < V; ++j) {
                double s = 0.0;
                for (int i = 0; i < K; ++i) s += H[IDX2(i, j, V)] * qt[i];
                yt[j] = s + wrn[j] * vt[j];
            }
            if (states)
                memcpy(states + (IDX2(b, n, N) * (size_t)(T + 1) + (size_t)(t + 1)) * KV, H,
                       KV * sizeof(double));
        }
        if (HT) memcpy(HT + IDX2(b, n, N) * KV, H, KV * sizeof(double));
        free(H); free(Hn); free(Z);
    }
    return err;
}

/* Backward pass (BPTT).  Every output is overwritten.  H0, dHT and dH0 may
 * be NULL.  dq and dk are summed over heads, dW and dw_r over batch and time. */
int m2rnn_oracle_bwd(int B, int T, int N, int K, int V,
                     const double *q, const double *k, const double *v,
                     const double *f, const double *W, const double *w_r,
                     const double *H0, const double *dy, const double *dHT,
                     double *dq, double *dk, double *dv, double *df,
                     double *dW, double *dw_r, double *dH0)
{
    if (B < 0 || T < 0 || N < 0 || K <= 0 || V <= 0) return -1;
    const size_t KV = (size_t)K * V;
    const size_t VV = (size_t)V * V;
    /* Per-(b, n) partial sums, reduced serially after the parallel loop. */
    double *dq_part = (double *)calloc((size_t)B * N * T * K + 1, sizeof(double));
    double *dk_part = (double *)calloc((size_t)B * N * T * K + 1, sizeof(double));
    double *dW_part = (double *)calloc((size_t)B * N * VV + 1, sizeof(double));
    double *dwr_part = (double *)calloc((size_t)B * N * V + 1, sizeof(double));
    if (!dq_part || !dk_part || !dW_part || !dwr_part) {
        free(dq_part); free(dk_part); free(dW_part); free(dwr_part);
        return -2;
    }
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bn = 0; bn < (long)B * N; ++bn) {
        const int b = (int)(bn / N), n = (int)(bn % N);
        /* All states H_0..H_T and all candidates Z_1..Z_T, kept in fp64. */
        double *Hs = (double *)malloc((size_t)(T + 1) * KV * sizeof(double));
        double *Zs = (double *)malloc(((size_t)T + 1) * KV * sizeof(double));
        double *C = (double *)malloc(KV * sizeof(double));
        double *R = (double *)malloc(KV * sizeof(double));
        double *D = (double *)malloc(KV * sizeof(double));
        if (!Hs || !Zs || !C || !R || !D) {
#pragma omp atomic write
            err = -2;
            free(Hs); free(Zs); free(C); free(R); free(D);
            continue;
        }
        const double *Wn = W + (size_t)n * VV;
        const double *wrn = w_r + (size_t)n * V;
        /* Recompute the trajectory. */
        if (H0) memcpy(Hs, H0 + IDX2(b, n, N) * KV, KV * sizeof(double));
        else memset(Hs, 0, KV * sizeof(double));
        for (int t = 0; t < T; ++t) {
            const double *kt = k + IDX2(b, t, T) * K;
            const double *vt = v + (IDX2(b, t, T) * N + n) * V;
            const double ft = f[IDX2(b, t, T) * N + n];
            oracle_step(K, V, Hs + (size_t)t * KV, Wn, kt, vt, ft,
                        Zs + (size_t)(t + 1) * KV, Hs + (size_t)(t + 1) * KV);
        }
        /* Reverse sweep.  Array step t (0-based) is the paper's step t+1:
         * it reads H_prev = Hs[t], writes H_cur = Hs[t+1], candidate Zs[t+1]. */
        if (dHT) memcpy(C, dHT + IDX2(b, n, N) * KV, KV * sizeof(double));
        else memset(C, 0, KV * sizeof(double));
        double *dWp = dW_part + (size_t)bn * VV;
        double *dwrp = dwr_part + (size_t)bn * V;
        for (int t = T - 1; t >= 0; --t) {
            const double *qt = q + IDX2(b, t, T) * K;
            const double *kt = k + IDX2(b, t, T) * K;
            const double *vt = v + (IDX2(b, t, T) * N + n) * V;
            const double *ut = dy + (IDX2(b, t, T) * N + n) * V;
            const double ft = f[IDX2(b, t, T) * N + n];
            const double *Hp = Hs + (size_t)t * KV;
            const double *Hc = Hs + (size_t)(t + 1) * KV;
            const double *Zt = Zs + (size_t)(t + 1) * KV;
            /* R_t = C_t + q_t u_t^T */
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j)
                    R[IDX2(i, j, V)] = C[IDX2(i, j, V)] + qt[i] * ut[j];
            /* D_t = ((1 - f_t) R_t) (.) (1 - Z_t (.) Z_t) */
            for (size_t e = 0; e < KV; ++e)
                D[e] = ((1.0 - ft) * R[e]) * (1.0 - Zt[e] * Zt[e]);
            /* dL/df_t = <R_t, H_{t-1} - Z_t>_F */
            double dft = 0.0;
            for (size_t e = 0; e < KV; ++e) dft += R[e] * (Hp[e] - Zt[e]);
            df[IDX2(b, t, T) * N + n] = dft;
            /* dL/dW += H_{t-1}^T D_t */
            for (int l = 0; l < V; ++l)
                for (int j = 0; j < V; ++j) {
                    double s = 0.0;
                    for (int i = 0; i < K; ++i) s += Hp[IDX2(i, l, V)] * D[IDX2(i, j, V)];
                    dWp[IDX2(l, j, V)] += s;
                }
            /* dk_t (this head's share) = D_t v_t */
            double *dkp = dk_part + (IDX2(b, n, N) * (size_t)T + (size_t)t) * K;
            for (int i = 0; i < K; ++i) {
                double s = 0.0;
                for (int j = 0; j < V; ++j) s += D[IDX2(i, j, V)] * vt[j];
                dkp[i] = s;
            }
            /* dv_t = D_t^T k_t + w_r (.) u_t */
            double *dvt = dv + (IDX2(b, t, T) * N + n) * V;
            for (int j = 0; j < V; ++j) {
                double s = 0.0;
                for (int i = 0; i < K; ++i) s += D[IDX2(i, j, V)] * kt[i];
                dvt[j] = s + wrn[j] * ut[j];
            }
            /* dq_t (this head's share) = H_t u_t */
            double *dqp = dq_part + (IDX2(b, n, N) * (size_t)T + (size_t)t) * K;
            for (int i = 0; i < K; ++i) {
                double s = 0.0;
                for (int j = 0; j < V; ++j) s += Hc[IDX2(i, j, V)] * ut[j];
                dqp[i] = s;
            }
            /* dL/dw_r += u_t (.) v_t */
            for (int j = 0; j < V; ++j) dwrp[j] += ut[j] * vt[j];
            /* C_{t-1} = f_t R_t + D_t W^T */
            for (int i = 0; i < K; ++i)
                for (int l = 0; l < V; ++l) {
                    double s = 0.0;
                    for (int j = 0; j < V; ++j) s += D[IDX2(i, j, V)] * Wn[IDX2(l, j, V)];
                    C[IDX2(i, l, V)] = ft * R[IDX2(i, l, V)] + s;
                }
        }
        if (dH0) memcpy(dH0 + IDX2(b, n, N) * KV, C, KV * sizeof(double));
        free(Hs); free(Zs); free(C); free(R); free(D);
    }
    if (err == 0) {
        /* Head sums for the shared q, k; batch-and-time sums for W, w_r. */
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < T; ++t)
                for (int i = 0; i < K; ++i) {
                    double sq = 0.0, sk = 0.0;
                    for (int n = 0; n < N; ++n) {
                        const size_t o = (IDX2(b, n, N) * (size_t)T + (size_t)t) * K + i;
                        sq += dq_part[o];
                        sk += dk_part[o];
                    }
                    dq[IDX2(b, t, T) * K + i] = sq;
                    dk[IDX2(b, t, T) * K + i] = sk;
                }
        for (int n = 0; n < N; ++n) {
            for (size_t e = 0; e < VV; ++e) {
                double s = 0.0;
                for (int b = 0; b < B; ++b) s += dW_part[IDX2(b, n, N) * VV + e];
                dW[(size_t)n * VV + e] = s;
            }
            for (int j = 0; j < V; ++j) {
                double s = 0.0;
                for (int b = 0; b < B; ++b) s += dwr_part[IDX2(b, n, N) * V + j];
                dw_r[(size_t)n * V + j] = s;
            }
        }
    }
    free(dq_part); free(dk_part); free(dW_part); free(dwr_part);
    return err;
}
