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
 * Layouts: row-major; xhat, gy, dxhat [B,T,P]; a, u, c, h, mu [B,T,N];
 * W_a, W_B, W_c, dW_* [P,N]; W_o, dW_o [N,P]; b_a, db_a [N].  Tokens are stored
 * 0-based: array row t holds token t+1 of the pages' 1-based notation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_LITERAL 0
#define ORC_AGGREGATED 1

/* one layer forward, [AS] Assumptions (Sec. 3.1 SSM dynamics, Sec. 3.2 residual);
 * xres (the residual input) may be NULL, meaning xhat itself */
void orc_layer_forward(int64_t B, int64_t T, int64_t P, int64_t N,
                       const double *W_a, const double *W_B, const double *W_c,
                       const double *b_a, const double *W_o, const double *xhat, const double *xres,
                       double *a, double *u, double *c, double *h, double *y)
{
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < T; ++t) {
            const double *x = xhat + (b * T + t) * P;
            double *at = a + (b * T + t) * N, *ut = u + (b * T + t) * N;
            double *ct = c + (b * T + t) * N, *ht = h + (b * T + t) * N;
            const double *hprev = t > 0 ? h + (b * T + t - 1) * N : NULL;
            for (int64_t n = 0; n < N; ++n) {
                double za = b_a[n], zu = 0.0, zc = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    za += x[p] * W_a[p * N + n];
                    zu += x[p] * W_B[p * N + n];
                    zc += x[p] * W_c[p * N + n];
                }
                at[n] = 1.0 / (1.0 + exp(-za));
                ut[n] = zu;
                ct[n] = zc;
                ht[n] = at[n] * (hprev ? hprev[n] : 0.0) + ut[n];
            }
            double *yt = y + (b * T + t) * P;
            const double *xr = xres ? xres + (b * T + t) * P : x;
            for (int64_t p = 0; p < P; ++p) {
                double s = xr[p];
                for (int64_t n = 0; n < N; ++n) s += ct[n] * ht[n] * W_o[n * P + p];
                yt[p] = s;
            }
        }
    }
}

/* vjp^{A_i} and vjp^{B_i} of token i for the adjoint vector v (length N) */
static void vjp_AB(int64_t P, int64_t N, const double *W_a, const double *W_B,
                   const double *x, const double *a_i, const double *h_im1, const double *v,
                   double *s_scratch, double *dW_a, double *dW_B, double *db_a, double *dx)
{
    for (int64_t n = 0; n < N; ++n)
        s_scratch[n] = v[n] * (h_im1 ? h_im1[n] : 0.0) * a_i[n] * (1.0 - a_i[n]);
    for (int64_t n = 0; n < N; ++n) db_a[n] += s_scratch[n];
    for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            dW_a[p * N + n] += x[p] * s_scratch[n];
            dW_B[p * N + n] += x[p] * v[n];
            acc += s_scratch[n] * W_a[p * N + n] + v[n] * W_B[p * N + n];
        }
        dx[p] += acc;
    }
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

    double *g = malloc(sizeof(double) * N);
    double *v = malloc(sizeof(double) * N);
    double *s = malloc(sizeof(double) * N);
    double *V = mode == ORC_AGGREGATED ? calloc((size_t)(T * N), sizeof(double)) : NULL;
    int64_t count = 0;

    for (int64_t b = 0; b < B; ++b) {
        const double *xb = xhat + b * T * P, *gyb = gy + b * T * P;
        const double *ab = a + b * T * N, *cb = c + b * T * N, *hb = h + b * T * N;
        double *dxb = dxhat + b * T * P;
        double *mub = mu ? mu + b * T * N : NULL;
        if (V) memset(V, 0, sizeof(double) * T * N);

        for (int64_t t = 0; t < T; ++t) {
            /* g_t = gy_t W_o^T : the cotangent of (c_t . h_t) */
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t p = 0; p < P; ++p) acc += gyb[t * P + p] * W_o[n * P + p];
                g[n] = acc;
            }
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
            if (mode == ORC_LITERAL) {
                for (int64_t i = t; i >= lo; --i) {
                    for (int64_t n = 0; n < N; ++n) {
                        double prod = 1.0; /* prod_{j=i+1..t} a_j, explicit */
                        for (int64_t j = i + 1; j <= t; ++j) prod *= ab[j * N + n];
                        v[n] = g[n] * cb[t * N + n] * prod;
                        if (mub) mub[i * N + n] += v[n];
                    }
                    vjp_AB(P, N, W_a, W_B, xb + i * P, ab + i * N,
                           i > 0 ? hb + (i - 1) * N : NULL, v, s, dW_a, dW_B, db_a, dxb + i * P);
                    ++count;
                }
            } else {
                for (int64_t n = 0; n < N; ++n) v[n] = g[n] * cb[t * N + n];
                for (int64_t i = t; i >= lo; --i) {
                    for (int64_t n = 0; n < N; ++n) {
                        V[i * N + n] += v[n];
                        v[n] *= ab[i * N + n]; /* v_{t,i-1} = v_{t,i} . a_i */
                    }
                    ++count;
                }
            }
        }
        if (mode == ORC_AGGREGATED) {
            for (int64_t i = 0; i < T; ++i) {
                vjp_AB(P, N, W_a, W_B, xb + i * P, ab + i * N,
                       i > 0 ? hb + (i - 1) * N : NULL, V + i * N, s, dW_a, dW_B, db_a, dxb + i * P);
                if (mub) memcpy(mub + i * N, V + i * N, sizeof(double) * N);
            }
        }
    }
    free(g); free(v); free(s); free(V);
    return count;
}
