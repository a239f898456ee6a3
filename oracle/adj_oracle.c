/*
 * adj_oracle.c -- plain, slow, fp64 CPU oracle for the adjoint-sharding gradient
 * of one diagonal selective SSM layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) includes, links or calls this file; only the tests, the
 * smoke check and the benchmark's CPU-baseline leg do.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * Source: the review page "Adjoint sharding for very long context training of
 * state space models" (pith.science), cited below as [AS] with the part of the
 * page the formula comes from.  Model, in the diagonal selective form:
 *
 *   a_t = sigmoid(xhat_t W_a + b_a), u_t = xhat_t W_B, c_t = xhat_t W_c     ([AS] Assumptions, Sec. 3.1)
 *   h_t = a_t . h_{t-1} + u_t,  h_0 = 0   (A_t = diag(a_t), B_t xhat_t = u_t)
 *   ytilde_t = (c_t . h_t) W_o            (C_t = W_o^T diag(c_t))
 *   y_t = xres_t + ytilde_t               ([AS] What carries the argument, residual identity;
 *                                          xres = y^{k-1}, the residual stream entering the layer)
 *
 * Gradient ([AS] Core claim, Proposition 2), for a cotangent gy_t = dL/dy_t:
 *
 *   dl_t/dtheta = sum_{i<=t} vjp^{A_i}(dl_t/dy_t lambda_{t,i} (x) h_{i-1})
 *               + sum_{i<=t} vjp^{B_i}(dl_t/dy_t lambda_{t,i} (x) xhat_i)
 *               + vjp^{C_t}(dl_t/dy_t (x) h_t)
 *   lambda_{t,i} = C_t prod_{j=i+1..t} A_j          ([AS] What carries the argument)
 *
 * so that dl_t/dy_t lambda_{t,i} = g_t . c_t . prod_{j=i+1..t} a_j with
 * g_t = gy_t W_o^T.  Truncated adjoint sharding ([AS] Core claim, last sentence;
 * Referee Report, Section 4.3) keeps only the pairs with t - i < Tbar.
 *
 * The VJPs written out (sigma'(z) = a(1-a)):
 *   vjp^{A_i}(v (x) h_{i-1}): s = v . h_{i-1} . a_i . (1-a_i);
 *                             dW_a += xhat_i^T s, db_a += s, dxhat_i += s W_a^T
 *   vjp^{B_i}(v (x) xhat_i):  dW_B += xhat_i^T v, dxhat_i += v W_B^T
 *   vjp^{C_t}(gy_t (x) h_t):  dW_o += (c_t . h_t)^T gy_t;
 *                             dW_c += xhat_t^T (g_t . h_t), dxhat_t += (g_t . h_t) W_c^T
 *
 * Two evaluation modes, both summing every (t,i) pair:
 *   ORC_LITERAL:    each lambda product is formed by explicit multiplication and
 *                   each VJP is applied on its own (O(T^2 (T N + P N))).
 *   ORC_AGGREGATED: each pair's adjoint vector v_{t,i} is still formed (walking i
 *                   down from t, v_{t,i-1} = v_{t,i} . a_i), but the VJPs of one
 *                   token i are applied once to V_i = sum_t v_{t,i}; exact by the
 *                   linearity of a VJP in its seed vector (O(T Tbar N + T P N)).
 *
 * Threads: the aggregated mode and the forward pass run their loops over tokens,
 * channels or rows of the weight gradients in parallel (OpenMP, when compiled with
 * it).  Every output element is still computed by one thread with its sums taken in
 * the same order as a plain serial loop over b, t (and p or n), so the results do not
 * depend on the thread count.  The literal mode is serial.
 *
 * Layouts: row-major; xhat, gy, dxhat [B,T,P]; a, u, c, h, mu [B,T,N];
 * W_a, W_B, W_c, dW_* [P,N]; W_o, dW_o [N,P]; b_a, db_a [N].  Tokens are stored
 * 0-based: array row t holds token t+1 of the pages' 1-based notation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_LITERAL 0
#define ORC_AGGREGATED 1

/* Set the number of threads of the parallel loops (n > 0) and return the number in use
 * (1 when built without OpenMP). */
int orc_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Rows [*lo, *hi) of n rows owned by the calling thread (all rows without OpenMP). */
static void thread_rows(int64_t n, int64_t *lo, int64_t *hi)
{
#ifdef _OPENMP
    const int64_t k = omp_get_thread_num(), m = omp_get_num_threads();
    *lo = n * k / m;
    *hi = n * (k + 1) / m;
#else
    *lo = 0;
    *hi = n;
#endif
}

#define ORC_TB 8   /* tokens per block of the weight-sweeping loops (each weight row is reused) */

/* one layer forward, [AS] Assumptions (Sec. 3.1 SSM dynamics, Sec. 3.2 residual);
 * xres (the residual input) may be NULL, meaning xhat itself */
void orc_layer_forward(int64_t B, int64_t T, int64_t P, int64_t N,
                       const double *W_a, const double *W_B, const double *W_c,
                       const double *b_a, const double *W_o, const double *xhat, const double *xres,
                       double *a, double *u, double *c, double *h, double *y)
{
    const int64_t BT = B * T;
    /* a_t, u_t, c_t of every token: each pre-activation summed over p in order */
#pragma omp parallel for schedule(static)
    for (int64_t r0 = 0; r0 < BT; r0 += ORC_TB) {
        const int64_t r1 = r0 + ORC_TB < BT ? r0 + ORC_TB : BT;
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t n = 0; n < N; ++n) {
                a[r * N + n] = b_a[n];
                u[r * N + n] = 0.0;
                c[r * N + n] = 0.0;
            }
        for (int64_t p = 0; p < P; ++p) {
            const double *wa = W_a + p * N, *wb = W_B + p * N, *wc = W_c + p * N;
            for (int64_t r = r0; r < r1; ++r) {
                const double xp = xhat[r * P + p];
                double *at = a + r * N, *ut = u + r * N, *ct = c + r * N;
                for (int64_t n = 0; n < N; ++n) {
                    at[n] += xp * wa[n];
                    ut[n] += xp * wb[n];
                    ct[n] += xp * wc[n];
                }
            }
        }
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t n = 0; n < N; ++n) a[r * N + n] = 1.0 / (1.0 + exp(-a[r * N + n]));
    }
    /* h_t = a_t . h_{t-1} + u_t, one channel of one sequence at a time */
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t t = 0; t < T; ++t) {
                const double *at = a + (b * T + t) * N, *ut = u + (b * T + t) * N;
                double *ht = h + (b * T + t) * N;
                const double *hprev = t > 0 ? h + (b * T + t - 1) * N : NULL;
                ht[n] = at[n] * (hprev ? hprev[n] : 0.0) + ut[n];
            }
        }
    }
    /* y_t = xres_t + (c_t . h_t) W_o, each output summed over n in order */
#pragma omp parallel for schedule(static)
    for (int64_t r0 = 0; r0 < BT; r0 += ORC_TB) {
        const int64_t r1 = r0 + ORC_TB < BT ? r0 + ORC_TB : BT;
        for (int64_t r = r0; r < r1; ++r) {
            const double *xr = xres ? xres + r * P : xhat + r * P;
            for (int64_t p = 0; p < P; ++p) y[r * P + p] = xr[p];
        }
        for (int64_t n = 0; n < N; ++n) {
            const double *wo = W_o + n * P;
            for (int64_t r = r0; r < r1; ++r) {
                const double chn = c[r * N + n] * h[r * N + n];
                double *yt = y + r * P;
                for (int64_t p = 0; p < P; ++p) yt[p] += chn * wo[p];
            }
        }
    }
}

/* g_t = gy_t W_o^T, the cotangent of (c_t . h_t), for tokens t0 <= t < t1 of one
 * sequence (g holds one row of N per token, from t0) */
static void cot_g(int64_t P, int64_t N, const double *W_o, const double *gyb, int64_t t0, int64_t t1, double *g)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t t = t0; t < t1; ++t) {
            double acc = 0.0;
            for (int64_t p = 0; p < P; ++p) acc += gyb[t * P + p] * W_o[n * P + p];
            g[(t - t0) * N + n] = acc;
        }
}

/* the A_i seed s = v . h_{i-1} . sigma'(z_i), sigma'(z) = a (1 - a) */
static void seed_A(int64_t N, const double *v, const double *h_im1, const double *a_i, double *s_scratch)
{
    for (int64_t n = 0; n < N; ++n)
        s_scratch[n] = v[n] * (h_im1 ? h_im1[n] : 0.0) * a_i[n] * (1.0 - a_i[n]);
}

/* the input part of vjp^{A_i} and vjp^{B_i} for nt consecutive tokens (rows of N in
 * s_all and v_all, rows of P in dx): dx += s W_a^T + v W_B^T */
static void vjp_AB_dx(int64_t P, int64_t N, const double *W_a, const double *W_B,
                      const double *s_all, const double *v_all, int64_t nt, double *dx)
{
    for (int64_t p = 0; p < P; ++p)
        for (int64_t j = 0; j < nt; ++j) {
            const double *s_scratch = s_all + j * N, *v = v_all + j * N;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n)
                acc += s_scratch[n] * W_a[p * N + n] + v[n] * W_B[p * N + n];
            dx[j * P + p] += acc;
        }
}

/* vjp^{A_i} and vjp^{B_i} of token i for the adjoint vector v (length N) */
static void vjp_AB(int64_t P, int64_t N, const double *W_a, const double *W_B,
                   const double *x, const double *a_i, const double *h_im1, const double *v,
                   double *s_scratch, double *dW_a, double *dW_B, double *db_a, double *dx)
{
    seed_A(N, v, h_im1, a_i, s_scratch);
    for (int64_t n = 0; n < N; ++n) db_a[n] += s_scratch[n];
    for (int64_t p = 0; p < P; ++p) {
        for (int64_t n = 0; n < N; ++n) {
            dW_a[p * N + n] += x[p] * s_scratch[n];
            dW_B[p * N + n] += x[p] * v[n];
        }
    }
    vjp_AB_dx(P, N, W_a, W_B, s_scratch, v, 1, dx);
}

/* Literal mode: every pair (t, i) with its own explicit product and its own VJP. */
static void grad_literal(int64_t B, int64_t T, int64_t P, int64_t N, int64_t Tbar,
                         const double *W_a, const double *W_B, const double *W_c,
                         const double *W_o, const double *xhat, const double *a,
                         const double *c, const double *h, const double *gy,
                         double *dW_a, double *dW_B, double *dW_c, double *db_a, double *dW_o,
                         double *dxhat, double *mu)
{
    double *g = malloc(sizeof(double) * N);
    double *v = malloc(sizeof(double) * N);
    double *s = malloc(sizeof(double) * N);
    for (int64_t b = 0; b < B; ++b) {
        const double *xb = xhat + b * T * P, *gyb = gy + b * T * P;
        const double *ab = a + b * T * N, *cb = c + b * T * N, *hb = h + b * T * N;
        double *dxb = dxhat + b * T * P;
        double *mub = mu ? mu + b * T * N : NULL;
        for (int64_t t = 0; t < T; ++t) {
            cot_g(P, N, W_o, gyb, t, t + 1, g);
            /* vjp^{C_t}(dl_t/dy_t (x) h_t) */
            for (int64_t n = 0; n < N; ++n)
                for (int64_t p = 0; p < P; ++p)
                    dW_o[n * P + p] += cb[t * N + n] * hb[t * N + n] * gyb[t * P + p];
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double gh = g[n] * hb[t * N + n];
                    dW_c[p * N + n] += xb[t * P + p] * gh;
                    acc += gh * W_c[p * N + n];
                }
                dxb[t * P + p] += acc;
            }
            /* the pairs (t, i), i = t, t-1, ..., t-Tbar+1 (0-based rows) */
            int64_t lo = t - Tbar + 1;
            if (lo < 0) lo = 0;
            for (int64_t i = t; i >= lo; --i) {
                for (int64_t n = 0; n < N; ++n) {
                    double prod = 1.0; /* prod_{j=i+1..t} a_j, explicit */
                    for (int64_t j = i + 1; j <= t; ++j) prod *= ab[j * N + n];
                    v[n] = g[n] * cb[t * N + n] * prod;
                    if (mub) mub[i * N + n] += v[n];
                }
                vjp_AB(P, N, W_a, W_B, xb + i * P, ab + i * N,
                       i > 0 ? hb + (i - 1) * N : NULL, v, s, dW_a, dW_B, db_a, dxb + i * P);
            }
        }
    }
    free(g); free(v); free(s);
}

/* Aggregated mode, in phases over all tokens.  Each phase splits its work over outputs
 * that are disjoint between threads and keeps, for every output element, the summation
 * order of the serial loop over b, t: the same values as a serial evaluation. */
static void grad_aggregated(int64_t B, int64_t T, int64_t P, int64_t N, int64_t Tbar,
                            const double *W_a, const double *W_B, const double *W_c,
                            const double *W_o, const double *xhat, const double *a,
                            const double *c, const double *h, const double *gy,
                            double *dW_a, double *dW_B, double *dW_c, double *db_a, double *dW_o,
                            double *dxhat, double *mu)
{
    const int64_t BT = B * T;
    double *G = malloc(sizeof(double) * BT * N);       /* g_t of every token */
    double *Vall = calloc((size_t)(BT * N), sizeof(double));   /* V_i = sum_t v_{t,i} */
    double *Sall = malloc(sizeof(double) * BT * N);    /* A_i seeds of V_i */

    /* g_t = gy_t W_o^T, blocks of tokens within one sequence */
    const int64_t TBLK = (T + ORC_TB - 1) / ORC_TB;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t q = 0; q < TBLK; ++q) {
            const int64_t t0 = q * ORC_TB, t1 = t0 + ORC_TB < T ? t0 + ORC_TB : T;
            cot_g(P, N, W_o, gy + b * T * P, t0, t1, G + (b * T + t0) * N);
        }

    /* vjp^{C_t}(dl_t/dy_t (x) h_t): dW_o rows and dW_c rows split between threads, every
     * token's row read once per thread; dxhat by blocks of tokens */
#pragma omp parallel
    {
        int64_t n0, n1, p0, p1;
        thread_rows(N, &n0, &n1);
        for (int64_t r = 0; r < BT; ++r)
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t p = 0; p < P; ++p)
                    dW_o[n * P + p] += c[r * N + n] * h[r * N + n] * gy[r * P + p];
        thread_rows(P, &p0, &p1);
        for (int64_t r = 0; r < BT; ++r)
            for (int64_t p = p0; p < p1; ++p)
                for (int64_t n = 0; n < N; ++n)
                    dW_c[p * N + n] += xhat[r * P + p] * (G[r * N + n] * h[r * N + n]);
    }
#pragma omp parallel for schedule(static)
    for (int64_t r0 = 0; r0 < BT; r0 += ORC_TB) {
        const int64_t r1 = r0 + ORC_TB < BT ? r0 + ORC_TB : BT;
        for (int64_t p = 0; p < P; ++p)
            for (int64_t r = r0; r < r1; ++r) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += (G[r * N + n] * h[r * N + n]) * W_c[p * N + n];
                dxhat[r * P + p] += acc;
            }
    }

    /* every pair (t, i), t - Tbar < i <= t: v_{t,i} formed by walking i down from t
     * (v_{t,t} = g_t . c_t, v_{t,i-1} = v_{t,i} . a_i) and added into V_i.  One thread
     * owns one sequence and a group of 8 channels, copied to contiguous scratch. */
    const int64_t NG = (N + 7) / 8;
#pragma omp parallel
    {
        double *v = malloc(sizeof(double) * N);
        double *Vg = malloc(sizeof(double) * T * 8), *ag = malloc(sizeof(double) * T * 8);
#pragma omp for collapse(2) schedule(dynamic)
        for (int64_t b = 0; b < B; ++b) {
            for (int64_t q = 0; q < NG; ++q) {
                const int64_t n0 = q * 8, n1 = n0 + 8 < N ? n0 + 8 : N, w = n1 - n0;
                const double *cb = c + b * T * N, *g = G + b * T * N;
                double *V = Vg - n0;                        /* V[i * 8 + n], n0 <= n < n1 */
                const double *ab = ag - n0;
                for (int64_t i = 0; i < T; ++i)
                    for (int64_t k = 0; k < w; ++k) {
                        ag[i * 8 + k] = a[(b * T + i) * N + n0 + k];
                        Vg[i * 8 + k] = 0.0;
                    }
                for (int64_t t = 0; t < T; ++t) {
                    int64_t lo = t - Tbar + 1;
                    if (lo < 0) lo = 0;
                    for (int64_t n = n0; n < n1; ++n) v[n] = g[t * N + n] * cb[t * N + n];
                    for (int64_t i = t; i >= lo; --i) {
                        for (int64_t n = n0; n < n1; ++n) {
                            V[i * 8 + n] += v[n];
                            v[n] *= ab[i * 8 + n]; /* v_{t,i-1} = v_{t,i} . a_i */
                        }
                    }
                }
                for (int64_t i = 0; i < T; ++i)
                    for (int64_t k = 0; k < w; ++k) Vall[(b * T + i) * N + n0 + k] = Vg[i * 8 + k];
            }
        }
        free(v); free(Vg); free(ag);
    }

    /* vjp^{A_i} and vjp^{B_i}, once per token on V_i */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < BT; ++r) {
        const int64_t b = r / T, i = r % T;
        const double *hb = h + b * T * N;
        seed_A(N, Vall + r * N, i > 0 ? hb + (i - 1) * N : NULL, a + r * N, Sall + r * N);
    }
#pragma omp parallel
    {
        int64_t n0, n1, p0, p1;
        thread_rows(N, &n0, &n1);
        for (int64_t r = 0; r < BT; ++r) {
            const double *s_scratch = Sall + r * N;
            for (int64_t n = n0; n < n1; ++n) db_a[n] += s_scratch[n];
        }
        thread_rows(P, &p0, &p1);
        for (int64_t r = 0; r < BT; ++r)
            for (int64_t p = p0; p < p1; ++p) {
                const double xp = xhat[r * P + p];
                for (int64_t n = 0; n < N; ++n) {
                    dW_a[p * N + n] += xp * Sall[r * N + n];
                    dW_B[p * N + n] += xp * Vall[r * N + n];
                }
            }
    }
#pragma omp parallel for schedule(static)
    for (int64_t r0 = 0; r0 < BT; r0 += ORC_TB) {
        const int64_t r1 = r0 + ORC_TB < BT ? r0 + ORC_TB : BT;
        vjp_AB_dx(P, N, W_a, W_B, Sall + r0 * N, Vall + r0 * N, r1 - r0, dxhat + r0 * P);
    }
    if (mu) memcpy(mu, Vall, sizeof(double) * BT * N);
    free(G); free(Vall); free(Sall);
}

/*
 * Gradient of one layer for the cotangent gy = dL/dy ([AS] Core claim,
 * Proposition 2; Proposition 3 applies it per layer with that layer's total
 * cotangent).  Tbar <= 0 means the full adjoint; otherwise only pairs with
 * t - i < Tbar.  Outputs are overwritten.  dxhat receives dL/dxhat through this
 * layer's A, B, C paths only (the residual identity adds gy on top).  mu, if not
 * NULL, receives V_i = sum_t dl_t/dy_t lambda_{t,i}.  Returns the number of
 * (t,i) VJP pairs evaluated.
 */
int64_t orc_layer_grad(int64_t B, int64_t T, int64_t P, int64_t N, int64_t Tbar, int mode,
                       const double *W_a, const double *W_B, const double *W_c,
                       const double *W_o, const double *xhat, const double *a,
                       const double *c, const double *h, const double *gy,
                       double *dW_a, double *dW_B, double *dW_c, double *db_a, double *dW_o,
                       double *dxhat, double *mu)
{
    memset(dW_a, 0, sizeof(double) * P * N);
    memset(dW_B, 0, sizeof(double) * P * N);
    memset(dW_c, 0, sizeof(double) * P * N);
    memset(db_a, 0, sizeof(double) * N);
    memset(dW_o, 0, sizeof(double) * N * P);
    memset(dxhat, 0, sizeof(double) * B * T * P);
    if (mu) memset(mu, 0, sizeof(double) * B * T * N);
    if (Tbar <= 0 || Tbar > T) Tbar = T;

    int64_t count = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < T; ++t) {
            int64_t lo = t - Tbar + 1;
            if (lo < 0) lo = 0;
            count += t - lo + 1;
        }
    if (mode == ORC_LITERAL)
        grad_literal(B, T, P, N, Tbar, W_a, W_B, W_c, W_o, xhat, a, c, h, gy,
                     dW_a, dW_B, dW_c, db_a, dW_o, dxhat, mu);
    else
        grad_aggregated(B, T, P, N, Tbar, W_a, W_B, W_c, W_o, xhat, a, c, h, gy,
                        dW_a, dW_B, dW_c, db_a, dW_o, dxhat, mu);
    return count;
}
