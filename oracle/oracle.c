/*
 * oracle.c -- plain float64 CPU reference for the linear-recurrence hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links or calls this file;
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark do.
 * It shares no code, header, helper or constant with the CUDA sources.
 *
 * Every function is the plain definition, written as a sequential loop in
 * float64, one independent unit (a batch row and channel, or a batch row and
 * head) at a time.  OpenMP only splits those independent units across cores;
 * it never reorders the arithmetic inside a unit.
 *
 * Sources (page title, section):
 *   "Parallel Scan" (zerotofrontier.app/ssm/parallel-scan), sections
 *     "The scan for one number of state", "Scans over vector and matrix
 *     states", "What one combine costs", "A vectorized scan for diagonal
 *     states", "The backward pass is a scan in reverse", "The backward pass of
 *     linear attention", "The chunkwise algorithm", "When a scan is the wrong
 *     tool".
 *   "Lightning Attention-2" (paper-graph-ui, arXiv 2401.04658), eq. 4
 *     (recurrent form kv_t = lambda kv_{t-1} + k_t^T v_t, o_t = q_t kv_t) and
 *     eqs. 11-12 (per-token gradients).
 *
 * Layouts (row-major, innermost last):
 *   diagonal scan:    a, b, h, g, da, db        [B][T][D];  h0, hT, dhT, dh0 [B][D]
 *   selective scan:   x, delta, y, dy, dx, ddelta [B][T][D]; A, dA [D][N];
 *                     Bm, Cm, dB, dC [B][T][N];  h0, hT, dhT, dh0 [B][D][N]
 *   linear attention: q, k, dq, dk [B][H][T][dk]; v, o, dO, dv [B][H][T][dv];
 *                     log_a, dlog_a [B][H][T];   S0, ST, dST, dS0 [B][H][dk][dv]
 *   gated (GLA):      as linear attention, with log_a, dlog_a [B][H][T][dk]
 * Optional pointers may be NULL (meaning zero for inputs, "not wanted" for
 * outputs).  Time indices below are 1-based in comments (t = 1..T), matching
 * the pages, and 0-based in code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Diagonal scan, forward.                                                   */
/* "Parallel Scan", "The scan for one number of state": h_t = a_t h_{t-1} +  */
/* b_t, h_0 = 0 unless given; "A vectorized scan for diagonal states": the   */
/* diagonal case is D independent scalar recurrences side by side.          */
/* ------------------------------------------------------------------------ */
void oracle_scan_diag_fwd(const double *a, const double *b, const double *h0,
                          double *h, double *hT, i64 B, i64 T, i64 D) {
    i64 units = B * D;
#pragma omp parallel for schedule(static)
    for (i64 u = 0; u < units; ++u) {
        i64 bi = u / D, d = u % D;
        double state = h0 ? h0[bi * D + d] : 0.0;
        for (i64 t = 0; t < T; ++t) {
            i64 idx = (bi * T + t) * D + d;
            state = a[idx] * state + b[idx];
            h[idx] = state;
        }
        if (hT) hT[bi * D + d] = state;
    }
}

/* ------------------------------------------------------------------------ */
/* Diagonal scan, backward.                                                  */
/* "Parallel Scan", "The backward pass is a scan in reverse": with direct    */
/* gradients g_t = dL/dh_t, the adjoint obeys hbar_T = g_T and              */
/* hbar_t = g_t + a_{t+1} hbar_{t+1}; then dL/db_t = hbar_t,                 */
/* dL/da_t = hbar_t h_{t-1}, dL/dh_0 = a_1 hbar_1.  An optional gradient on  */
/* the returned final state (dhT) is one more direct gradient on h_T.        */
/* The states h_t are recomputed here from (a, b, h0) by the forward loop.   */
/* ------------------------------------------------------------------------ */
void oracle_scan_diag_bwd(const double *a, const double *b, const double *h0,
                          const double *g, const double *dhT, double *da,
                          double *db, double *dh0, i64 B, i64 T, i64 D) {
    i64 units = B * D;
#pragma omp parallel
    {
        double *hs = (double *)malloc(sizeof(double) * (size_t)(T + 1));
#pragma omp for schedule(static)
        for (i64 u = 0; u < units; ++u) {
            i64 bi = u / D, d = u % D;
            /* hs[t] holds h_t for t = 0..T (1-based time). */
            hs[0] = h0 ? h0[bi * D + d] : 0.0;
            for (i64 t = 1; t <= T; ++t) {
                i64 idx = (bi * T + (t - 1)) * D + d;
                hs[t] = a[idx] * hs[t - 1] + b[idx];
            }
            double hbar = 0.0;
            double a_next = 0.0; /* a_{t+1}; unused at t = T */
            for (i64 t = T; t >= 1; --t) {
                i64 idx = (bi * T + (t - 1)) * D + d;
                if (t == T)
                    hbar = g[idx] + (dhT ? dhT[bi * D + d] : 0.0);
                else
                    hbar = g[idx] + a_next * hbar;
                db[idx] = hbar;
                da[idx] = hbar * hs[t - 1];
                a_next = a[idx];
            }
            if (dh0) dh0[bi * D + d] = (T > 0) ? a_next * hbar : 0.0;
        }
        free(hs);
    }
}

/* ------------------------------------------------------------------------ */
/* Selective (Mamba-1 style) diagonal scan, forward.                         */
/* "Parallel Scan", "Scans over vector and matrix states" and "When a scan   */
/* is the wrong tool": every channel d keeps N state numbers, each with its  */
/* own decay a_{t,d,n} = exp(Delta_{t,d} A_{d,n}); the input written is      */
/* b_{t,d,n} = Delta_{t,d} B_t[n] x_{t,d}; the read is y_{t,d} =             */
/* sum_n C_t[n] h_{t,d,n}.  Each (d, n) is one scalar recurrence.            */
/* ------------------------------------------------------------------------ */
void oracle_selective_fwd(const double *x, const double *delta, const double *A,
                          const double *Bm, const double *Cm, const double *h0,
                          double *y, double *hT, i64 B, i64 T, i64 D, i64 N) {
    i64 units = B * D;
#pragma omp parallel
    {
        double *hs = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(static)
        for (i64 u = 0; u < units; ++u) {
            i64 bi = u / D, d = u % D;
            for (i64 n = 0; n < N; ++n)
                hs[n] = h0 ? h0[(bi * D + d) * N + n] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                i64 idx = (bi * T + t) * D + d;
                const double *Bt = Bm + (bi * T + t) * N;
                const double *Ct = Cm + (bi * T + t) * N;
                double acc = 0.0;
                for (i64 n = 0; n < N; ++n) {
                    double a_tn = exp(delta[idx] * A[d * N + n]);
                    double b_tn = delta[idx] * Bt[n] * x[idx];
                    hs[n] = a_tn * hs[n] + b_tn;
                    acc += Ct[n] * hs[n];
                }
                y[idx] = acc;
            }
            if (hT)
                for (i64 n = 0; n < N; ++n) hT[(bi * D + d) * N + n] = hs[n];
        }
        free(hs);
    }
}

/* ------------------------------------------------------------------------ */
/* Selective scan, backward: the adjoint recurrence of the diagonal scan      */
/* applied per (d, n) with direct gradient g_{t,d,n} = C_t[n] dy_{t,d}, then  */
/* the chain rule through a = exp(Delta A) and b = Delta B x:                 */
/*   dx_{t,d}     = sum_n hbar Delta B_t[n]                                   */
/*   dDelta_{t,d} = sum_n (hbar h_{t-1} a A_{d,n} + hbar B_t[n] x)            */
/*   dA_{d,n}     = sum_{b,t} hbar h_{t-1} a Delta                            */
/*   dB_t[n]      = sum_d hbar Delta x,      dC_t[n] = sum_d dy h_t           */
/*   dh0          = a_1 hbar_1                                               */
/* ------------------------------------------------------------------------ */
void oracle_selective_bwd(const double *x, const double *delta, const double *A,
                          const double *Bm, const double *Cm, const double *h0,
                          const double *dy, const double *dhT, double *dx,
                          double *ddelta, double *dA, double *dBm, double *dCm,
                          double *dh0, i64 B, i64 T, i64 D, i64 N) {
    i64 units = B * D;
    int nthr = oracle_num_threads();
    /* dB and dC are sums over channels: each thread accumulates the channels
       it owns into a private [B][T][N] array; the arrays are then added in
       thread order.  dA sums over batch and time: kept per (b, d), added over
       b afterwards. */
    double *accB = (double *)calloc((size_t)nthr * (size_t)(B * T * N), sizeof(double));
    double *accC = (double *)calloc((size_t)nthr * (size_t)(B * T * N), sizeof(double));
    double *pdA = (double *)calloc((size_t)(B * D * N), sizeof(double));
#pragma omp parallel num_threads(nthr)
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *myB = accB + (size_t)tid * (size_t)(B * T * N);
        double *myC = accC + (size_t)tid * (size_t)(B * T * N);
        double *hs = (double *)malloc(sizeof(double) * (size_t)((T + 1) * N));
        double *hbar = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(static)
        for (i64 u = 0; u < units; ++u) {
            i64 bi = u / D, d = u % D;
            /* forward recompute: hs[t*N + n] = h_{t,n}, t = 0..T */
            for (i64 n = 0; n < N; ++n)
                hs[n] = h0 ? h0[(bi * D + d) * N + n] : 0.0;
            for (i64 t = 1; t <= T; ++t) {
                i64 idx = (bi * T + (t - 1)) * D + d;
                const double *Bt = Bm + (bi * T + (t - 1)) * N;
                for (i64 n = 0; n < N; ++n) {
                    double a_tn = exp(delta[idx] * A[d * N + n]);
                    double b_tn = delta[idx] * Bt[n] * x[idx];
                    hs[t * N + n] = a_tn * hs[(t - 1) * N + n] + b_tn;
                }
            }
            double *pa = pdA + (bi * D + d) * N;
            for (i64 t = T; t >= 1; --t) {
                i64 idx = (bi * T + (t - 1)) * D + d;
                const double *Bt = Bm + (bi * T + (t - 1)) * N;
                const double *Ct = Cm + (bi * T + (t - 1)) * N;
                double gx = 0.0, gdelta = 0.0;
                double *pB = myB + (bi * T + (t - 1)) * N;
                double *pC = myC + (bi * T + (t - 1)) * N;
                for (i64 n = 0; n < N; ++n) {
                    double g = Ct[n] * dy[idx];
                    if (t == T) {
                        hbar[n] = g + (dhT ? dhT[(bi * D + d) * N + n] : 0.0);
                    } else {
                        i64 idx1 = (bi * T + t) * D + d; /* step t+1 */
                        double a_next = exp(delta[idx1] * A[d * N + n]);
                        hbar[n] = g + a_next * hbar[n];
                    }
                    double a_tn = exp(delta[idx] * A[d * N + n]);
                    double h_prev = hs[(t - 1) * N + n];
                    double dadecay = hbar[n] * h_prev; /* dL/da_t */
                    gx += hbar[n] * delta[idx] * Bt[n];
                    gdelta += dadecay * a_tn * A[d * N + n] + hbar[n] * Bt[n] * x[idx];
                    pa[n] += dadecay * a_tn * delta[idx];
                    pB[n] += hbar[n] * delta[idx] * x[idx];
                    pC[n] += dy[idx] * hs[t * N + n];
                }
                dx[idx] = gx;
                ddelta[idx] = gdelta;
            }
            if (dh0) {
                for (i64 n = 0; n < N; ++n) {
                    double a1 = (T > 0) ? exp(delta[(bi * T) * D + d] * A[d * N + n]) : 0.0;
                    dh0[(bi * D + d) * N + n] = (T > 0) ? a1 * hbar[n] : 0.0;
                }
            }
        }
        free(hs);
        free(hbar);
    }
    for (i64 i = 0; i < B * T * N; ++i) {
        double sB = 0.0, sC = 0.0;
        for (int th = 0; th < nthr; ++th) {
            sB += accB[(size_t)th * (size_t)(B * T * N) + (size_t)i];
            sC += accC[(size_t)th * (size_t)(B * T * N) + (size_t)i];
        }
        dBm[i] = sB;
        dCm[i] = sC;
    }
    if (dA) {
        for (i64 d = 0; d < D; ++d)
            for (i64 n = 0; n < N; ++n) {
                double s = 0.0;
                for (i64 bi = 0; bi < B; ++bi) s += pdA[(bi * D + d) * N + n];
                dA[d * N + n] = s;
            }
    }
    free(accB);
    free(accC);
    free(pdA);
}

/* ------------------------------------------------------------------------ */
/* Decayed linear attention, forward, as its per-token recurrence.           */
/* "Parallel Scan", "The chunkwise algorithm": S_t = a_t S_{t-1} + k_t v_t^T */
/* (rows of S indexed by keys), update first, then read o_t = S_t^T q_t;     */
/* S_0 given.  The chunkwise algorithm reaches exactly these outputs up to    */
/* rounding, so this loop is the definition it is checked against.           */
/* "Lightning Attention-2", eq. 4, is the constant-decay special case.       */
/* ------------------------------------------------------------------------ */
void oracle_la_fwd(const double *q, const double *k, const double *v,
                   const double *log_a, const double *S0, double *o, double *ST,
                   i64 B, i64 H, i64 T, i64 dk, i64 dv) {
    i64 units = B * H;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
#pragma omp for schedule(static)
        for (i64 u = 0; u < units; ++u) {
            for (i64 i = 0; i < dk * dv; ++i) S[i] = S0 ? S0[u * dk * dv + i] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                const double *qt = q + (u * T + t) * dk;
                const double *kt = k + (u * T + t) * dk;
                const double *vt = v + (u * T + t) * dv;
                double at = exp(log_a[u * T + t]);
                for (i64 i = 0; i < dk; ++i)
                    for (i64 j = 0; j < dv; ++j)
                        S[i * dv + j] = at * S[i * dv + j] + kt[i] * vt[j];
                double *ot = o + (u * T + t) * dv;
                for (i64 j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (i64 i = 0; i < dk; ++i) s += S[i * dv + j] * qt[i];
                    ot[j] = s;
                }
            }
            if (ST)
                for (i64 i = 0; i < dk * dv; ++i) ST[u * dk * dv + i] = S[i];
        }
        free(S);
    }
}

/* ------------------------------------------------------------------------ */
/* Decayed linear attention, backward, by its definition.                    */
/* "Parallel Scan", "The backward pass of linear attention": the adjoint     */
/* state obeys Sbar_t = q_t obar_t^T + a_{t+1} Sbar_{t+1} (plus dS_T at      */
/* t = T), and                                                               */
/*   dq_t = S_t obar_t        (forward sweep: needs the forward state)       */
/*   dk_t = Sbar_t v_t,  dv_t = Sbar_t^T k_t                                 */
/*   dL/da_t = <Sbar_t, S_{t-1}>, so dL/dlog a_t = a_t <Sbar_t, S_{t-1}>      */
/*   dS_0 = a_1 Sbar_1.                                                      */
/* S_{t-1} is needed in the reverse sweep; it is recomputed block by block   */
/* from stored checkpoints (every CKPT steps) with the same forward loop, so */
/* the values are identical to a run that kept every state.                 */
/* ------------------------------------------------------------------------ */
#define ORACLE_LA_CKPT 64
void oracle_la_bwd(const double *q, const double *k, const double *v,
                   const double *log_a, const double *S0, const double *dO,
                   const double *dST, double *dq, double *dkk, double *dvv,
                   double *dlog_a, double *dS0, i64 B, i64 H, i64 T, i64 dk,
                   i64 dv) {
    i64 units = B * H;
    i64 nblk = (T + ORACLE_LA_CKPT - 1) / ORACLE_LA_CKPT;
    i64 ss = dk * dv;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)ss);
        double *Sbar = (double *)malloc(sizeof(double) * (size_t)ss);
        /* ckpt[b] = S at the start of block b (state S_{b*CKPT}) */
        double *ckpt = (double *)malloc(sizeof(double) * (size_t)((nblk + 1) * ss));
        /* blk[r] = S_{t0 + r} for r = 0..CKPT within the current block */
        double *blk = (double *)malloc(sizeof(double) * (size_t)((ORACLE_LA_CKPT + 1) * ss));
#pragma omp for schedule(static)
        for (i64 u = 0; u < units; ++u) {
            const double *qu = q + u * T * dk, *ku = k + u * T * dk;
            const double *vu = v + u * T * dv, *du = dO + u * T * dv;
            const double *lu = log_a + u * T;
            /* forward sweep: checkpoints and dq_t = S_t obar_t */
            for (i64 i = 0; i < ss; ++i) S[i] = S0 ? S0[u * ss + i] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                if (t % ORACLE_LA_CKPT == 0) memcpy(ckpt + (t / ORACLE_LA_CKPT) * ss, S, sizeof(double) * (size_t)ss);
                double at = exp(lu[t]);
                for (i64 i = 0; i < dk; ++i)
                    for (i64 j = 0; j < dv; ++j)
                        S[i * dv + j] = at * S[i * dv + j] + ku[t * dk + i] * vu[t * dv + j];
                for (i64 i = 0; i < dk; ++i) {
                    double s = 0.0;
                    for (i64 j = 0; j < dv; ++j) s += S[i * dv + j] * du[t * dv + j];
                    dq[(u * T + t) * dk + i] = s;
                }
            }
            /* reverse sweep */
            for (i64 i = 0; i < ss; ++i) Sbar[i] = dST ? dST[u * ss + i] : 0.0;
            double a_next = 1.0; /* a_{t+1}; the dS_T term enters undecayed */
            for (i64 bk = nblk - 1; bk >= 0; --bk) {
                i64 t0 = bk * ORACLE_LA_CKPT;
                i64 t1 = t0 + ORACLE_LA_CKPT < T ? t0 + ORACLE_LA_CKPT : T;
                memcpy(blk, ckpt + bk * ss, sizeof(double) * (size_t)ss);
                for (i64 t = t0; t < t1; ++t) {
                    double at = exp(lu[t]);
                    double *prev = blk + (t - t0) * ss, *cur = blk + (t - t0 + 1) * ss;
                    for (i64 i = 0; i < dk; ++i)
                        for (i64 j = 0; j < dv; ++j)
                            cur[i * dv + j] = at * prev[i * dv + j] + ku[t * dk + i] * vu[t * dv + j];
                }
                for (i64 t = t1 - 1; t >= t0; --t) {
                    /* Sbar_t = q_t obar_t^T + a_{t+1} Sbar_{t+1} */
                    for (i64 i = 0; i < dk; ++i)
                        for (i64 j = 0; j < dv; ++j)
                            Sbar[i * dv + j] = a_next * Sbar[i * dv + j] + qu[t * dk + i] * du[t * dv + j];
                    for (i64 i = 0; i < dk; ++i) {
                        double s = 0.0;
                        for (i64 j = 0; j < dv; ++j) s += Sbar[i * dv + j] * vu[t * dv + j];
                        dkk[(u * T + t) * dk + i] = s;
                    }
                    for (i64 j = 0; j < dv; ++j) {
                        double s = 0.0;
                        for (i64 i = 0; i < dk; ++i) s += Sbar[i * dv + j] * ku[t * dk + i];
                        dvv[(u * T + t) * dv + j] = s;
                    }
                    double at = exp(lu[t]);
                    if (dlog_a) {
                        const double *Sprev = blk + (t - t0) * ss;
                        double s = 0.0;
                        for (i64 i = 0; i < ss; ++i) s += Sbar[i] * Sprev[i];
                        dlog_a[u * T + t] = at * s;
                    }
                    a_next = at;
                }
            }
            if (dS0)
                for (i64 i = 0; i < ss; ++i) dS0[u * ss + i] = (T > 0 ? a_next : 1.0) * Sbar[i];
        }
        free(S);
        free(Sbar);
        free(ckpt);
        free(blk);
    }
}

/* ------------------------------------------------------------------------ */
/* Closed-form decay gradient ("Parallel Scan", "The backward pass of linear */
/* attention", the theorem after the four per-step gradients): with dq, dk   */
/* the full query and key gradients,                                         */
/*   dL/dlog a_u = sum_{t>=u} q_t.dq_t - sum_{s>=u} k_s.dk_s  (+ <dS_T,S_T>)  */
/* The last term is this library's reading for a gradient arriving on the   */
/* returned final state; the page's derivation has none.  It needs no        */
/* states.  Used to pin the definition above, and as a property at sizes the */
/* definition is too slow for.                                               */
/* ------------------------------------------------------------------------ */
void oracle_la_dlog_closed_form(const double *q, const double *k,
                                const double *dq, const double *dkk,
                                const double *dST, const double *ST,
                                double *dlog_a, i64 B, i64 H, i64 T, i64 dk,
                                i64 dv) {
    i64 units = B * H;
#pragma omp parallel for schedule(static)
    for (i64 u = 0; u < units; ++u) {
        double tail = 0.0;
        if (dST && ST)
            for (i64 i = 0; i < dk * dv; ++i) tail += dST[u * dk * dv + i] * ST[u * dk * dv + i];
        double run = tail;
        for (i64 t = T - 1; t >= 0; --t) {
            double qd = 0.0, kd = 0.0;
            for (i64 i = 0; i < dk; ++i) {
                qd += q[(u * T + t) * dk + i] * dq[(u * T + t) * dk + i];
                kd += k[(u * T + t) * dk + i] * dkk[(u * T + t) * dk + i];
            }
            run += qd - kd;
            dlog_a[u * T + t] = run;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Gated linear attention: one decay per key dimension.                     */
/* "Parallel Scan", "What one combine costs" (a diagonal transition, one    */
/* decay per state entry: GLA) and "The chunkwise algorithm" (the GLA form  */
/* S_t = G_t (.) S_{t-1} + k_t^T v_t, o_t = q_t S_t, G_t holding the        */
/* decays): here G_t[i][j] = a_t[i], one decay per key dimension i.         */
/*   log_a, dlog_a [B][H][T][dk]; other layouts as for linear attention.    */
/* ------------------------------------------------------------------------ */
void oracle_gla_fwd(const double *q, const double *k, const double *v,
                    const double *log_a, const double *S0, double *o, double *ST,
                    i64 B, i64 H, i64 T, i64 dk, i64 dv) {
    i64 units = B * H;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
#pragma omp for schedule(static)
        for (i64 u = 0; u < units; ++u) {
            for (i64 i = 0; i < dk * dv; ++i) S[i] = S0 ? S0[u * dk * dv + i] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                const double *qt = q + (u * T + t) * dk;
                const double *kt = k + (u * T + t) * dk;
                const double *vt = v + (u * T + t) * dv;
                const double *lt = log_a + (u * T + t) * dk;
                for (i64 i = 0; i < dk; ++i) {
                    double ai = exp(lt[i]);
                    for (i64 j = 0; j < dv; ++j) S[i * dv + j] = ai * S[i * dv + j] + kt[i] * vt[j];
                }
                double *ot = o + (u * T + t) * dv;
                for (i64 j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (i64 i = 0; i < dk; ++i) s += S[i * dv + j] * qt[i];
                    ot[j] = s;
                }
            }
            if (ST)
                for (i64 i = 0; i < dk * dv; ++i) ST[u * dk * dv + i] = S[i];
        }
        free(S);
    }
}

/* Backward by the adjoint definition ("Parallel Scan", "The backward pass of */
/* linear attention", with the scalar decay replaced by the diagonal one):    */
/*   Sbar_t = q_t^T obar_t + diag(a_{t+1}) Sbar_{t+1}  (+ dS_T at t = T)      */
/*   dq_t = S_t obar_t,  dk_t = Sbar_t v_t,  dv_t = Sbar_t^T k_t              */
/*   dL/dlog a_t[i] = a_t[i] sum_j Sbar_t[i][j] S_{t-1}[i][j]                 */
/*   dS_0 = diag(a_1) Sbar_1.                                                 */
/* Every forward state is kept (the oracle runs on short sequences only).    */
void oracle_gla_bwd(const double *q, const double *k, const double *v,
                    const double *log_a, const double *S0, const double *dO,
                    const double *dST, double *dq, double *dkk, double *dvv,
                    double *dlog_a, double *dS0, i64 B, i64 H, i64 T, i64 dk,
                    i64 dv) {
    i64 units = B * H;
    i64 ss = dk * dv;
#pragma omp parallel
    {
        double *states = (double *)malloc(sizeof(double) * (size_t)((T + 1) * ss)); /* S_0..S_T */
        double *Sbar = (double *)malloc(sizeof(double) * (size_t)ss);
        double *anext = (double *)malloc(sizeof(double) * (size_t)dk);
#pragma omp for schedule(static)
        for (i64 u = 0; u < units; ++u) {
            const double *qu = q + u * T * dk, *ku = k + u * T * dk;
            const double *vu = v + u * T * dv, *du = dO + u * T * dv;
            const double *lu = log_a + u * T * dk;
            for (i64 i = 0; i < ss; ++i) states[i] = S0 ? S0[u * ss + i] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                const double *prev = states + t * ss;
                double *cur = states + (t + 1) * ss;
                for (i64 i = 0; i < dk; ++i) {
                    double ai = exp(lu[t * dk + i]);
                    for (i64 j = 0; j < dv; ++j) cur[i * dv + j] = ai * prev[i * dv + j] + ku[t * dk + i] * vu[t * dv + j];
                }
                for (i64 i = 0; i < dk; ++i) {
                    double s = 0.0;
                    for (i64 j = 0; j < dv; ++j) s += cur[i * dv + j] * du[t * dv + j];
                    dq[(u * T + t) * dk + i] = s;
                }
            }
            for (i64 i = 0; i < ss; ++i) Sbar[i] = dST ? dST[u * ss + i] : 0.0;
            for (i64 i = 0; i < dk; ++i) anext[i] = 1.0; /* the dS_T term enters undecayed */
            for (i64 t = T - 1; t >= 0; --t) {
                for (i64 i = 0; i < dk; ++i)
                    for (i64 j = 0; j < dv; ++j)
                        Sbar[i * dv + j] = anext[i] * Sbar[i * dv + j] + qu[t * dk + i] * du[t * dv + j];
                for (i64 i = 0; i < dk; ++i) {
                    double s = 0.0;
                    for (i64 j = 0; j < dv; ++j) s += Sbar[i * dv + j] * vu[t * dv + j];
                    dkk[(u * T + t) * dk + i] = s;
                }
                for (i64 j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (i64 i = 0; i < dk; ++i) s += Sbar[i * dv + j] * ku[t * dk + i];
                    dvv[(u * T + t) * dv + j] = s;
                }
                const double *Sprev = states + t * ss;
                for (i64 i = 0; i < dk; ++i) {
                    double ai = exp(lu[t * dk + i]);
                    if (dlog_a) {
                        double s = 0.0;
                        for (i64 j = 0; j < dv; ++j) s += Sbar[i * dv + j] * Sprev[i * dv + j];
                        dlog_a[(u * T + t) * dk + i] = ai * s;
                    }
                    anext[i] = ai;
                }
            }
            if (dS0)
                for (i64 i = 0; i < dk; ++i)
                    for (i64 j = 0; j < dv; ++j) dS0[u * ss + i * dv + j] = anext[i] * Sbar[i * dv + j];
        }
        free(states);
        free(Sbar);
        free(anext);
    }
}

/* Closed-form decay gradient per key dimension ("Parallel Scan", "The        */
/* backward pass of linear attention": the closed form there is Yang et al.'s */
/* for gated linear attention, one decay per key dimension): path by path,    */
/* a contribution through key dimension i crosses step u exactly when its    */
/* write is before u and its read at or after u, so                           */
/*   dL/dlog a_u[i] = sum_{t>=u} q_t[i] dq_t[i] - sum_{s>=u} k_s[i] dk_s[i]   */
/*                    (+ sum_j dS_T[i][j] S_T[i][j]).                          */
void oracle_gla_dlog_closed_form(const double *q, const double *k,
                                 const double *dq, const double *dkk,
                                 const double *dST, const double *ST,
                                 double *dlog_a, i64 B, i64 H, i64 T, i64 dk,
                                 i64 dv) {
    i64 units = B * H;
#pragma omp parallel for schedule(static)
    for (i64 u = 0; u < units; ++u) {
        for (i64 i = 0; i < dk; ++i) {
            double run = 0.0;
            if (dST && ST)
                for (i64 j = 0; j < dv; ++j) run += dST[u * dk * dv + i * dv + j] * ST[u * dk * dv + i * dv + j];
            for (i64 t = T - 1; t >= 0; --t) {
                i64 x = (u * T + t) * dk + i;
                run += q[x] * dq[x] - k[x] * dkk[x];
                dlog_a[x] = run;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* State passing between slices of one sequence ("Parallel Scan", "Splitting */
/* one sequence across devices"): a slice run from a zero state gives its   */
/* pair (alpha, dS): its total decay and its own contribution to its final  */
/* state.  The state entering a later slice is the earlier pairs composed    */
/* under (a1, b1) . (a2, b2) = (a1 a2, a2 b1 + b2) and applied to the       */
/* initial state ("The scan for one number of state": the combine), i.e.    */
/* the fold acc <- alpha_j acc + dS_j over the pairs in order.               */
/*   decay_total: alpha[bh][a] = exp(sum_t log_decay[bh][t][a])              */
/*   state_compose: pairs j = first + c * step, c = 0..count-1; alpha       */
/*   [P][BH][A] (A = 1: one decay per head; A = rows: one per state row),    */
/*   dS [P][BH][n], edge [BH][n] or NULL, out [BH][n].                       */
/* ------------------------------------------------------------------------ */
void oracle_decay_total(const double *log_decay, double *alpha, i64 BH, i64 T, i64 A) {
    for (i64 bh = 0; bh < BH; ++bh)
        for (i64 a = 0; a < A; ++a) {
            double s = 0.0;
            for (i64 t = 0; t < T; ++t) s += log_decay[(bh * T + t) * A + a];
            alpha[bh * A + a] = exp(s);
        }
}

void oracle_state_compose(const double *alpha, const double *dS, const double *edge, double *out,
                          i64 P, i64 BH, i64 n, i64 A, i64 first, i64 count, i64 step) {
    (void)P;
    i64 per = n / A;
    for (i64 bh = 0; bh < BH; ++bh)
        for (i64 e = 0; e < n; ++e) {
            double acc = edge ? edge[bh * n + e] : 0.0;
            for (i64 c = 0; c < count; ++c) {
                i64 j = first + c * step;
                acc = alpha[(j * BH + bh) * A + e / per] * acc + dS[(j * BH + bh) * n + e];
            }
            out[bh * n + e] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Delta rule with a decay per head (Gated DeltaNet).  "Parallel Scan",     */
/* "What one combine costs": the transition is the identity minus a rank-   */
/* one matrix, and the write overwrites what the state stores under a key   */
/* instead of only adding to it; "At real scale": the Gated DeltaNet layer  */
/* has a scalar decay per head besides.  In the pages' row convention       */
/* (S [dk][dv], rows indexed by keys, o_t = q_t S_t):                       */
/*   S_t = a_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t            */
/* with a_t = exp(log_a_t) per (head, token) and beta_t per (head, token):  */
/* with beta = 1 and a unit key, k_t S_t = v_t -- the value now stored      */
/* under k_t is exactly v_t.                                                 */
/*   q, k [B][H][T][dk]; v [B][H][T][dv]; log_a, beta [B][H][T];           */
/*   S0, ST [B][H][dk][dv].                                                  */
/* ------------------------------------------------------------------------ */
static void delta_step(const double *kt, const double *vt, double at, double bt, const double *prev,
                       double *cur, double *u, i64 dk, i64 dv) {
    /* u = k_t S_{t-1} (the value stored under k_t before the write) */
    for (i64 j = 0; j < dv; ++j) {
        double s = 0.0;
        for (i64 i = 0; i < dk; ++i) s += kt[i] * prev[i * dv + j];
        u[j] = s;
    }
    for (i64 i = 0; i < dk; ++i)
        for (i64 j = 0; j < dv; ++j)
            cur[i * dv + j] = at * (prev[i * dv + j] - bt * kt[i] * u[j]) + bt * kt[i] * vt[j];
}

void oracle_delta_fwd(const double *q, const double *k, const double *v, const double *log_a,
                      const double *beta, const double *S0, double *o, double *ST, i64 B, i64 H,
                      i64 T, i64 dk, i64 dv) {
    i64 units = B * H, ss = dk * dv;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)ss);
        double *N = (double *)malloc(sizeof(double) * (size_t)ss);
        double *u = (double *)malloc(sizeof(double) * (size_t)dv);
#pragma omp for schedule(static)
        for (i64 un = 0; un < units; ++un) {
            for (i64 i = 0; i < ss; ++i) S[i] = S0 ? S0[un * ss + i] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                const double *qt = q + (un * T + t) * dk;
                delta_step(k + (un * T + t) * dk, v + (un * T + t) * dv, exp(log_a[un * T + t]),
                           beta[un * T + t], S, N, u, dk, dv);
                for (i64 i = 0; i < ss; ++i) S[i] = N[i];
                for (i64 j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (i64 i = 0; i < dk; ++i) s += qt[i] * S[i * dv + j];
                    o[(un * T + t) * dv + j] = s;
                }
            }
            if (ST)
                for (i64 i = 0; i < ss; ++i) ST[un * ss + i] = S[i];
        }
        free(S);
        free(N);
        free(u);
    }
}

/* Backward by the adjoint.  With M_t = a_t (I - beta_t k_t^T k_t)           */
/* (symmetric), u_t = k_t S_{t-1} and Sbar_t = dL/dS_t:                      */
/*   Sbar_t = q_t^T obar_t + M_{t+1} Sbar_{t+1}   (+ dST at t = T)           */
/*   dq_t = obar_t S_t^T                                                     */
/*   dv_t = beta_t k_t Sbar_t                                                */
/*   dbeta_t = (k_t Sbar_t) . (v_t - a_t u_t)                                */
/*   dk_t[m] = beta_t Sbar_t[m] . (v_t - a_t u_t)                            */
/*             - a_t beta_t S_{t-1}[m] . (k_t Sbar_t)                        */
/*   dlog a_t = <Sbar_t, M_t S_{t-1}>,   dS0 = M_1 Sbar_1.                   */
/* Every state is kept (short sequences only).                               */
void oracle_delta_bwd(const double *q, const double *k, const double *v, const double *log_a,
                      const double *beta, const double *S0, const double *dO, const double *dST,
                      double *dq, double *dkk, double *dvv, double *dlog_a, double *dbeta,
                      double *dS0, i64 B, i64 H, i64 T, i64 dk, i64 dv) {
    i64 units = B * H, ss = dk * dv;
#pragma omp parallel
    {
        double *states = (double *)malloc(sizeof(double) * (size_t)((T + 1) * ss));
        double *Sbar = (double *)malloc(sizeof(double) * (size_t)ss);
        double *tmp = (double *)malloc(sizeof(double) * (size_t)ss);
        double *u = (double *)malloc(sizeof(double) * (size_t)dv);
        double *kS = (double *)malloc(sizeof(double) * (size_t)dv);
#pragma omp for schedule(static)
        for (i64 un = 0; un < units; ++un) {
            const double *qu = q + un * T * dk, *ku = k + un * T * dk;
            const double *vu = v + un * T * dv, *du = dO + un * T * dv;
            for (i64 i = 0; i < ss; ++i) states[i] = S0 ? S0[un * ss + i] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                delta_step(ku + t * dk, vu + t * dv, exp(log_a[un * T + t]), beta[un * T + t],
                           states + t * ss, states + (t + 1) * ss, u, dk, dv);
                const double *cur = states + (t + 1) * ss;
                for (i64 i = 0; i < dk; ++i) {
                    double s = 0.0;
                    for (i64 j = 0; j < dv; ++j) s += cur[i * dv + j] * du[t * dv + j];
                    dq[(un * T + t) * dk + i] = s;
                }
            }
            for (i64 i = 0; i < ss; ++i) Sbar[i] = dST ? dST[un * ss + i] : 0.0;
            for (i64 t = T - 1; t >= 0; --t) {
                const double *kt = ku + t * dk, *vt = vu + t * dv, *qt = qu + t * dk;
                const double at = exp(log_a[un * T + t]), bt = beta[un * T + t];
                const double *prev = states + t * ss;
                /* Sbar_t: the later step's contribution is already in Sbar (M_{t+1} Sbar_{t+1}) */
                for (i64 i = 0; i < dk; ++i)
                    for (i64 j = 0; j < dv; ++j) Sbar[i * dv + j] += qt[i] * du[t * dv + j];
                for (i64 j = 0; j < dv; ++j) {
                    double su = 0.0, sk = 0.0;
                    for (i64 i = 0; i < dk; ++i) {
                        su += kt[i] * prev[i * dv + j];
                        sk += kt[i] * Sbar[i * dv + j];
                    }
                    u[j] = su;
                    kS[j] = sk;
                    dvv[(un * T + t) * dv + j] = bt * sk;
                }
                double db = 0.0;
                for (i64 j = 0; j < dv; ++j) db += kS[j] * (vt[j] - at * u[j]);
                if (dbeta) dbeta[un * T + t] = db;
                for (i64 m = 0; m < dk; ++m) {
                    double s1 = 0.0, s2 = 0.0;
                    for (i64 j = 0; j < dv; ++j) {
                        s1 += Sbar[m * dv + j] * (vt[j] - at * u[j]);
                        s2 += prev[m * dv + j] * kS[j];
                    }
                    dkk[(un * T + t) * dk + m] = bt * s1 - at * bt * s2;
                }
                if (dlog_a) {
                    /* <Sbar_t, M_t S_{t-1}> = a_t (<Sbar, S_{t-1}> - beta (k Sbar) . u) */
                    double s = 0.0;
                    for (i64 i = 0; i < ss; ++i) s += Sbar[i] * prev[i];
                    double c = 0.0;
                    for (i64 j = 0; j < dv; ++j) c += kS[j] * u[j];
                    dlog_a[un * T + t] = at * (s - bt * c);
                }
                /* Sbar <- M_t Sbar (the gradient on S_{t-1}) */
                for (i64 i = 0; i < dk; ++i)
                    for (i64 j = 0; j < dv; ++j) tmp[i * dv + j] = at * (Sbar[i * dv + j] - bt * kt[i] * kS[j]);
                for (i64 i = 0; i < ss; ++i) Sbar[i] = tmp[i];
            }
            if (dS0)
                for (i64 i = 0; i < ss; ++i) dS0[un * ss + i] = Sbar[i];
        }
        free(states);
        free(Sbar);
        free(tmp);
        free(u);
        free(kS);
    }
}
