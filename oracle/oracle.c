/*
 * CPU oracle for the Mamba-1 selective state-space scan.  TEST INFRASTRUCTURE ONLY:
 * the product path never links, loads or calls this file; only the tests, the smoke
 * check and the benchmark's CPU-baseline leg do.
 *
 * Everything is fp64 and strictly sequential in time.  No blocking, no fusion, no
 * reordering beyond the recurrence as the pages write it.  The only parallelism is
 * over independent (batch, channel) rows, which share no state.
 *
 * Sources (page address, section).  Two of the pages carry an unrelated site title, so the
 * pages are named by address:
 *  - Zero-order-hold discretisation, Abar = exp(dt A), Bbar = (dt A)^-1 (exp(dt A) - I) dt B:
 *    dpshk.com/news/3333417 section 2.2; lshu.cn/news/79586 section 2.2.  With diagonal A
 *    (S4D, dpshk.com/news/3333417 section 3.2) the matrix form becomes, per state n,
 *    Bbar = expm1(dt a_n) / a_n * b_n, whose a_n -> 0 limit is dt * b_n.
 *  - Simplified input matrix Bbar = dt * B: dpshk.com/news/3333417 sections 4.2 and 5.1.
 *  - Recurrence h_k = Abar h_{k-1} + Bbar x_k, y_k = C h_k + D x_k: dpshk.com/news/3333417
 *    sections 2.2 and 2.3 and the SelectiveSSM forward loop of section 5.1.
 *  - Selection dt = softplus(linear(x)): dpshk.com/news/3333417 section 4.1.
 *  - Causal depthwise conv1d (padding width-1, cropped to L) then SiLU, and the output
 *    gate y * SiLU(z): dpshk.com/news/3333417 section 5.2 (MambaBlock); lshu.cn/news/79586
 *    section 3.3.
 *  - Single-token step with the state carried as a cache: datadaily.news "State space
 *    models vs Transformer: a practical guide", section "how state space models work";
 *    lshu.cn/news/79586 section 6.5 (cache shape (batch, d_inner, d_state)).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_API __attribute__((visibility("default")))

static double softplus(double s) {
    /* log(1 + e^s), written so that neither branch overflows or cancels. */
    return s > 0.0 ? s + log1p(exp(-s)) : log1p(exp(s));
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* One scan problem description, shared by all worker threads. */
typedef struct {
    int R, L, N, W;
    const int *row_b, *row_d;
    const double *u, *delta, *z;          /* (R, L) each; z may be NULL            */
    const double *A;                      /* (D, N), indexed by the row's channel  */
    const double *Dskip, *delta_bias;     /* (D) or NULL                           */
    const double *conv_w, *conv_b;        /* (D, W), (D) or NULL                   */
    const double *Bm, *Cm;                /* (batch, N, L), indexed by row's batch */
    const double *h0;                     /* (R, N) or NULL                        */
    const double *conv_init;              /* (R, W-1): x before t = 0, or NULL     */
    double *conv_final;                   /* (R, W-1): the last W-1 x, or NULL     */
    double *y, *h_out;                    /* (R, L), (R, N) or NULL                */
    double *h_all;                        /* (R, L, N): the state after every step, or NULL */
    int delta_softplus, zoh;
    int next_row;                         /* work counter, guarded by lock         */
    pthread_mutex_t lock;
} scan_job;

static void scan_one_row(const scan_job *j, int r, double *h, double *v) {
    const int L = j->L, N = j->N, W = j->W;
    const int b = j->row_b[r], d = j->row_d[r];
    const double *ur = j->u + (size_t)r * L;
    const double *dr = j->delta + (size_t)r * L;
    const double *Ad = j->A + (size_t)d * N;
    const double *Bb = j->Bm + (size_t)b * N * L;
    const double *Cb = j->Cm + (size_t)b * N * L;

    /* Input to the SSM: the raw u, or SiLU(causal depthwise conv of x) when a conv is given.
       x before t = 0 is the row's conv_init history (oldest first) when given, else zero. */
    const double *xi = j->conv_init ? j->conv_init + (size_t)r * (W - 1) : NULL;
    for (int t = 0; t < L; ++t) {
        if (j->conv_w) {
            double acc = j->conv_b ? j->conv_b[d] : 0.0;
            for (int k = 0; k < W; ++k) {
                int src = t - (W - 1) + k;        /* tap k = W-1 multiplies x_t, tap 0 multiplies x_{t-W+1} */
                if (src >= 0) acc += j->conv_w[(size_t)d * W + k] * ur[src];
                else if (xi) acc += j->conv_w[(size_t)d * W + k] * xi[(W - 1) + src];
            }
            v[t] = silu(acc);
        } else {
            v[t] = ur[t];
        }
    }
    /* The conv history the next call needs: x_{L-W+1} .. x_{L-1}, reaching back into conv_init when
       L < W - 1.  Staged first: conv_final may be the same buffer as conv_init. */
    if (j->conv_w && j->conv_final && W > 1) {
        double hist[8];
        for (int i = 0; i < W - 1; ++i) {
            int t = L - (W - 1) + i;
            hist[i] = t >= 0 ? ur[t] : (xi ? xi[(W - 1) + t] : 0.0);
        }
        for (int i = 0; i < W - 1; ++i) j->conv_final[(size_t)r * (W - 1) + i] = hist[i];
    }

    for (int n = 0; n < N; ++n) h[n] = j->h0 ? j->h0[(size_t)r * N + n] : 0.0;

    for (int t = 0; t < L; ++t) {
        double s = dr[t] + (j->delta_bias ? j->delta_bias[d] : 0.0);
        double dt = j->delta_softplus ? softplus(s) : s;
        double y = 0.0;
        for (int n = 0; n < N; ++n) {
            double a = Ad[n];
            double Bt = Bb[(size_t)n * L + t];
            double Abar = exp(dt * a);
            double Bbar;
            if (j->zoh)
                Bbar = (a != 0.0 ? expm1(dt * a) / a : dt) * Bt;
            else
                Bbar = dt * Bt;
            h[n] = Abar * h[n] + Bbar * v[t];
            y += Cb[(size_t)n * L + t] * h[n];
            if (j->h_all) j->h_all[((size_t)r * L + t) * N + n] = h[n];
        }
        if (j->Dskip) y += j->Dskip[d] * v[t];
        if (j->z) y *= silu(j->z[(size_t)r * L + t]);
        j->y[(size_t)r * L + t] = y;
    }
    if (j->h_out)
        for (int n = 0; n < N; ++n) j->h_out[(size_t)r * N + n] = h[n];
}

static void *scan_worker(void *arg) {
    scan_job *j = (scan_job *)arg;
    double *h = (double *)malloc(sizeof(double) * (size_t)j->N);
    double *v = (double *)malloc(sizeof(double) * (size_t)(j->L > 0 ? j->L : 1));
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int r = j->next_row++;
        pthread_mutex_unlock(&j->lock);
        if (r >= j->R) break;
        scan_one_row(j, r, h, v);
    }
    free(h);
    free(v);
    return NULL;
}

static int resolve_threads(int nthreads, int R) {
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > R) nthreads = R > 0 ? R : 1;
    return nthreads;
}

/*
 * Selective scan over R independent rows.  Row r is (batch row_b[r], channel row_d[r]);
 * its u/delta/z/y are the r-th length-L rows of the compact (R, L) arrays, and its
 * initial/final state the r-th N-vector of h0/h_out.  h_all (R, L, N), when given, receives
 * the state after every step: the state sequence a multi-token verification pass keeps
 * (pwwt.cn/news/5168881 section 3.4).  Passing all (b, d) pairs in order
 * makes the compact layout equal to the full (B, D, L) layout.
 * Returns the number of threads used, or -1 on bad arguments.
 */
ORACLE_API int oracle_scan_rows(int R, int L, int N, const int *row_b, const int *row_d,
                                const double *u, const double *delta, const double *z,
                                const double *A, const double *Dskip, const double *delta_bias,
                                const double *conv_w, const double *conv_b, int conv_width,
                                const double *conv_init, double *conv_final,
                                const double *Bm, const double *Cm, const double *h0,
                                double *y, double *h_out, double *h_all, int delta_softplus, int zoh,
                                int nthreads) {
    if (R < 0 || L < 0 || N <= 0 || !row_b || !row_d || !u || !delta || !A || !Bm || !Cm || !y) return -1;
    if (conv_w && (conv_width <= 0 || conv_width > 8)) return -1;
    scan_job j;
    memset(&j, 0, sizeof(j));
    j.R = R; j.L = L; j.N = N; j.W = conv_width;
    j.row_b = row_b; j.row_d = row_d;
    j.u = u; j.delta = delta; j.z = z; j.A = A; j.Dskip = Dskip; j.delta_bias = delta_bias;
    j.conv_w = conv_w; j.conv_b = conv_b; j.Bm = Bm; j.Cm = Cm; j.h0 = h0; j.y = y; j.h_out = h_out;
    j.h_all = h_all;
    j.conv_init = conv_w ? conv_init : NULL;
    j.conv_final = conv_w ? conv_final : NULL;
    j.delta_softplus = delta_softplus; j.zoh = zoh;
    pthread_mutex_init(&j.lock, NULL);
    int nt = resolve_threads(nthreads, R);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, scan_worker, &j);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&j.lock);
    return nt;
}

/*
 * Causal depthwise conv1d over R rows of length L: out[t] = b + sum_k w[k] x[t-W+1+k]
 * (x before the row start is zero), optionally followed by SiLU.
 */
ORACLE_API int oracle_conv1d_rows(int R, int L, int W, const int *row_d, const double *x, const double *w,
                                  const double *b, int silu_on, double *out) {
    if (R < 0 || L < 0 || W <= 0 || !row_d || !x || !w || !out) return -1;
    for (int r = 0; r < R; ++r) {
        int d = row_d[r];
        const double *xr = x + (size_t)r * L;
        for (int t = 0; t < L; ++t) {
            double acc = b ? b[d] : 0.0;
            for (int k = 0; k < W; ++k) {
                int src = t - (W - 1) + k;
                if (src >= 0) acc += w[(size_t)d * W + k] * xr[src];
            }
            out[(size_t)r * L + t] = silu_on ? silu(acc) : acc;
        }
    }
    return 1;
}

/*
 * Single-token state update: the scan body with L = 1, starting from state (B, D, N)
 * and writing it back in place.  u, delta, z, y are (B, D); Bm, Cm are (B, N).
 * With conv_w given, u is the conv input x and conv_state (B, D, W-1) holds the previous W-1
 * inputs (oldest first): the step reads it as the conv history and leaves the last W-1 inputs
 * there (the decode cache's conv part: dpshk.com/news/5205047 section 1.3, lshu.cn/news/79586
 * section 6.5).
 */
ORACLE_API int oracle_state_update(int Bsz, int D, int N, double *state, const double *u, const double *delta,
                                   const double *A, const double *Bm, const double *Cm, const double *Dskip,
                                   const double *delta_bias, const double *z, const double *conv_w,
                                   const double *conv_b, int conv_width, double *conv_state, double *y,
                                   int delta_softplus, int zoh, int nthreads) {
    if (conv_w && !conv_state && conv_width > 1) return -1;
    if (Bsz < 0 || D < 0 || N <= 0 || !state || !u || !delta || !A || !Bm || !Cm || !y) return -1;
    int R = Bsz * D;
    int *rb = (int *)malloc(sizeof(int) * (size_t)(R > 0 ? R : 1));
    int *rd = (int *)malloc(sizeof(int) * (size_t)(R > 0 ? R : 1));
    for (int b = 0; b < Bsz; ++b)
        for (int d = 0; d < D; ++d) { rb[b * D + d] = b; rd[b * D + d] = d; }
    /* With L = 1 the (B, N, L) layout of Bm/Cm is exactly the (B, N) layout given here, and the
       state (B, D, N) is the compact (R, N) layout; scan_one_row copies h0 before it writes h_out,
       so passing the same buffer for both is safe. */
    int rc = oracle_scan_rows(R, 1, N, rb, rd, u, delta, z, A, Dskip, delta_bias, conv_w, conv_b, conv_width,
                              conv_state, conv_state, Bm, Cm, state, y, state, NULL, delta_softplus, zoh, nthreads);
    free(rb);
    free(rd);
    return rc;
}
