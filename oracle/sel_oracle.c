/*
 * sel_oracle.c -- plain, slow, fp64 CPU oracle for the adjoint-sharding gradient of one
 * general selective state-space layer (input-dependent A_t, B_t and C_t).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its Python
 * binding) includes, links or calls this file; only the tests and the smoke check do.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * Source: the review page "Adjoint sharding for very long context training of state
 * space models" (pith.science), cited as [AS].  The pages give the layer only in its
 * general form h_t = A_t h_{t-1} + B_t xhat_t, y_t = C_t h_t ([AS] Circularity Check,
 * assumptions; the derivation paragraph of the same check, Proposition 2), with A_t, B_t
 * and C_t functions of the token.  This file takes the plainest selective reading of that
 * form (stated once here and in the design notes), per channel p < P and state n < N:
 *
 *   z_t      = xhat_t W_in + [b_dt, 0, 0]       W_in = [W_dt | W_B | W_C], [P, P + 2N]
 *   dt_t,p   = softplus(z_t,p)                  step size of channel p
 *   B_t,n    = z_t,P+n,   C_t,n = z_t,P+N+n     input-dependent input and output maps
 *   Abar_t,pn = exp(dt_t,p A_pn)                A: [P, N], the continuous-time decay (< 0)
 *   h_t,pn   = Abar_t,pn h_t-1,pn + dt_t,p B_t,n xhat_t,p,   h_-1 = 0
 *   y_t,p    = xres_t,p + sum_n C_t,n h_t,pn    (residual identity, [AS] What carries the
 *                                                argument; xres = y^{k-1}, the residual stream
 *                                                entering the layer, xhat itself for a lone layer)
 *
 * In the pages' notation the state is the PN-vector h_t, A_t = diag(Abar_t) is diagonal,
 * B_t xhat_t = (dt_t,p B_t,n xhat_t,p)_pn, and C_t is the P x PN matrix with
 * C_t[p, (p,n)] = C_t,n: a full, input-dependent output map.
 *
 * Gradient ([AS] Core claim, Proposition 2), for a cotangent gy_t = dL/dy_t: the sum over
 * pairs (t, i <= t) of the VJP of step i applied to v_{t,i} = gy_t^T lambda_{t,i},
 * lambda_{t,i} = C_t prod_{j=i+1..t} A_j ([AS] What carries the argument), i.e.
 *
 *   v_{t,i},pn = gy_t,p C_t,n prod_{j=i+1..t} Abar_j,pn,
 *
 * plus the VJP of the output map at every token t.  Truncated adjoint sharding keeps the
 * pairs with t - i < Tbar ([AS] Core claim, last sentence).
 *
 * The VJPs written out, for a seed v on h_i (h_{i-1} held fixed, as the adjoint method
 * does):
 *   step i:   ddt_i,p += sum_n v_pn (A_pn Abar_i,pn h_{i-1},pn + B_i,n xhat_i,p)
 *             dA_pn   += v_pn dt_i,p Abar_i,pn h_{i-1},pn
 *             dB_i,n  += sum_p v_pn dt_i,p xhat_i,p
 *   output t: dC_t,n  += sum_p gy_t,p h_t,pn
 *   then      dz_i = [ddt_i . sigmoid(z_i,0..P-1) | dB_i | dC_i],
 *             dW_in += xhat_i^T dz_i,  db_dt += dz_i,0..P-1
 *   input path (for stacks, [AS] Core claim, Proposition 3):
 *             dxhat_i,p = sum_j dz_i,j W_in[p,j] + dt_i,p sum_n v_pn B_i,n
 *             (the projection, and xhat's own factor in the input term dt B xhat)
 *
 * Two evaluation modes, both summing every (t, i) pair in the window:
 *   literal:    every product prod_{j=i+1..t} Abar_j by explicit multiplication and every
 *               step VJP applied on its own (O(T^2 (T + P) P N));
 *   aggregated: every v_{t,i} still formed (walking i down from t, v_{t,i-1} = v_{t,i} .
 *               Abar_i), summed over t into V_i, and the step VJP applied once to V_i --
 *               exact by the linearity of a VJP in its seed (O(T Tbar P N + T P (P + 2N))).
 * Threads: the aggregated mode forms V in parallel over (b, p) (OpenMP when compiled with
 * it); every element keeps the serial summation order, so results do not depend on the
 * thread count.  The literal mode is serial.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double softplus(double z) { return z > 30.0 ? z : log1p(exp(z)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Forward pass.  x [B,T,P], xres [B,T,P] (NULL: x), W_in [P, P+2N], b_dt [P], A [P,N].
 * Writes z [B,T,P+2N] (with the bias), h [B,T,P,N], y [B,T,P]. */
void sel_forward(int64_t B, int64_t T, int64_t P, int64_t N, const double *x, const double *xres,
                 const double *W_in, const double *b_dt, const double *A, double *z, double *h, double *y)
{
    const int64_t Z = P + 2 * N;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t r = 0; r < B * T; ++r) {
        const double *xr = x + r * P;
        double *zr = z + r * Z;
        for (int64_t j = 0; j < Z; ++j) {
            double acc = 0.0;
            for (int64_t q = 0; q < P; ++q) acc += xr[q] * W_in[q * Z + j];
            zr[j] = acc + (j < P ? b_dt[j] : 0.0);
        }
    }
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < T; ++t) {
            const int64_t r = b * T + t;
            const double *zr = z + r * Z, *xr = x + r * P, *rr = (xres ? xres : x) + r * P;
            for (int64_t p = 0; p < P; ++p) {
                const double dt = softplus(zr[p]);
                double out = rr[p];
                for (int64_t n = 0; n < N; ++n) {
                    const double prev = t > 0 ? h[((r - 1) * P + p) * N + n] : 0.0;
                    const double hv = exp(dt * A[p * N + n]) * prev + dt * zr[P + n] * xr[p];
                    h[(r * P + p) * N + n] = hv;
                    out += zr[P + N + n] * hv;
                }
                y[r * P + p] = out;
            }
        }
    }
}

/* The VJP of step i (row r = b T + i) for the seed v [P,N]: adds into ddt [P] and dB [N]
 * of that row, and into dA [P,N]. */
static void vjp_step(int64_t P, int64_t N, const double *zr, const double *xr, const double *hprev,
                     const double *A, const double *v, double *ddt, double *dB, double *dA, double *dx)
{
    for (int64_t p = 0; p < P; ++p) {
        const double dt = softplus(zr[p]);
        for (int64_t n = 0; n < N; ++n) {
            const double ab = exp(dt * A[p * N + n]);
            const double hp = hprev ? hprev[p * N + n] : 0.0;
            const double vv = v[p * N + n];
            ddt[p] += vv * (A[p * N + n] * ab * hp + zr[P + n] * xr[p]);
            dA[p * N + n] += vv * dt * ab * hp;
            dB[n] += vv * dt * xr[p];
            if (dx) dx[p] += vv * dt * zr[P + n];
        }
    }
}

/* The output map's VJP at row r: dC [N] += sum_p gy_p h_pn. */
static void vjp_out(int64_t P, int64_t N, const double *gyr, const double *hr, double *dC)
{
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t p = 0; p < P; ++p) acc += gyr[p] * hr[p * N + n];
        dC[n] += acc;
    }
}

/* dz -> dW_in, db_dt (rows in order). */
static void param_from_dz(int64_t BT, int64_t P, int64_t N, const double *x, const double *dz,
                          double *dW_in, double *db_dt)
{
    const int64_t Z = P + 2 * N;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t q = 0; q < P; ++q)
        for (int64_t r = 0; r < BT; ++r) {
            const double xq = x[r * P + q];
            for (int64_t j = 0; j < Z; ++j) dW_in[q * Z + j] += xq * dz[r * Z + j];
        }
    for (int64_t r = 0; r < BT; ++r)
        for (int64_t p = 0; p < P; ++p) db_dt[p] += dz[r * Z + p];
}

static int64_t window_of(int64_t T, int64_t Tbar) { return (Tbar <= 0 || Tbar > T) ? T : Tbar; }

/* Gradient of one layer.  z, h from sel_forward; gy [B,T,P].  mode 0: literal, 1:
 * aggregated.  Writes (zeroing first) dz [B,T,P+2N], dW_in [P,P+2N], db_dt [P], dA [P,N],
 * if mu is not NULL mu [B,T,P,N] = sum over the window of v_{t,i}, and if dx is not NULL
 * the input path's cotangent dx [B,T,P] (not the residual's).  Returns the number of
 * (t, i) pairs summed per sequence. */
int64_t sel_grad(int64_t B, int64_t T, int64_t P, int64_t N, int64_t Tbar, int mode,
                 const double *x, const double *W_in, const double *A, const double *z, const double *h,
                 const double *gy, double *dz, double *dW_in, double *db_dt, double *dA, double *mu, double *dx)
{
    const int64_t Z = P + 2 * N, PN = P * N, W = window_of(T, Tbar);
    memset(dz, 0, sizeof(double) * (size_t)(B * T * Z));
    memset(dW_in, 0, sizeof(double) * (size_t)(P * Z));
    memset(db_dt, 0, sizeof(double) * (size_t)P);
    memset(dA, 0, sizeof(double) * (size_t)PN);
    if (mu) memset(mu, 0, sizeof(double) * (size_t)(B * T * PN));
    if (dx) memset(dx, 0, sizeof(double) * (size_t)(B * T * P));
    int64_t count = 0;
    for (int64_t t = 0; t < T; ++t) count += (t + 1 < W ? t + 1 : W);

    double *ddt = calloc((size_t)(B * T * P), sizeof(double));
    if (mode == 0) {
        double *v = malloc(sizeof(double) * (size_t)PN);
        for (int64_t b = 0; b < B; ++b)
            for (int64_t t = 0; t < T; ++t) {
                const int64_t rt = b * T + t;
                vjp_out(P, N, gy + rt * P, h + rt * PN, dz + rt * Z + P + N);
                int64_t lo = t - W + 1;
                if (lo < 0) lo = 0;
                for (int64_t i = t; i >= lo; --i) {
                    const int64_t ri = b * T + i;
                    for (int64_t p = 0; p < P; ++p)
                        for (int64_t n = 0; n < N; ++n) {
                            double prod = 1.0;   /* prod_{j=i+1..t} Abar_j, explicit */
                            for (int64_t j = i + 1; j <= t; ++j) {
                                const double dtj = softplus(z[(b * T + j) * Z + p]);
                                prod *= exp(dtj * A[p * N + n]);
                            }
                            v[p * N + n] = gy[rt * P + p] * z[rt * Z + P + N + n] * prod;
                            if (mu) mu[ri * PN + p * N + n] += v[p * N + n];
                        }
                    vjp_step(P, N, z + ri * Z, x + ri * P, i > 0 ? h + (ri - 1) * PN : NULL, A, v,
                             ddt + ri * P, dz + ri * Z + P, dA, dx ? dx + ri * P : NULL);
                }
            }
        free(v);
    } else {
        /* V_i = sum_{t=i}^{i+W-1} v_{t,i}, each pair's vector formed walking i down; the
         * factors Abar_i,pn = exp(dt_i,p A_pn) are tabulated once */
        double *V = calloc((size_t)(B * T * PN), sizeof(double));
        double *Ab = malloc(sizeof(double) * (size_t)(B * T * PN));
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t r = 0; r < B * T; ++r)
            for (int64_t p = 0; p < P; ++p) {
                const double dt = softplus(z[r * Z + p]);
                for (int64_t n = 0; n < N; ++n) Ab[r * PN + p * N + n] = exp(dt * A[p * N + n]);
            }
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
#endif
        for (int64_t b = 0; b < B; ++b)
            for (int64_t p = 0; p < P; ++p) {
                double *vv = malloc(sizeof(double) * (size_t)N);
                for (int64_t t = 0; t < T; ++t) {
                    const int64_t rt = b * T + t;
                    for (int64_t n = 0; n < N; ++n) vv[n] = gy[rt * P + p] * z[rt * Z + P + N + n];
                    int64_t lo = t - W + 1;
                    if (lo < 0) lo = 0;
                    for (int64_t i = t; i >= lo; --i) {
                        const int64_t ri = b * T + i;
                        double *Vi = V + ri * PN + p * N;
                        for (int64_t n = 0; n < N; ++n) Vi[n] += vv[n];
                        if (i > lo) {   /* v_{t,i-1} = v_{t,i} . Abar_i */
                            const double *ab = Ab + ri * PN + p * N;
                            for (int64_t n = 0; n < N; ++n) vv[n] *= ab[n];
                        }
                    }
                }
                free(vv);
            }
        free(Ab);
        for (int64_t b = 0; b < B; ++b)
            for (int64_t i = 0; i < T; ++i) {
                const int64_t ri = b * T + i;
                vjp_out(P, N, gy + ri * P, h + ri * PN, dz + ri * Z + P + N);
                vjp_step(P, N, z + ri * Z, x + ri * P, i > 0 ? h + (ri - 1) * PN : NULL, A, V + ri * PN,
                         ddt + ri * P, dz + ri * Z + P, dA, dx ? dx + ri * P : NULL);
            }
        if (mu) memcpy(mu, V, sizeof(double) * (size_t)(B * T * PN));
        free(V);
    }
    for (int64_t r = 0; r < B * T; ++r)
        for (int64_t p = 0; p < P; ++p) dz[r * Z + p] = ddt[r * P + p] * sigmoid(z[r * Z + p]);
    free(ddt);
    param_from_dz(B * T, P, N, x, dz, dW_in, db_dt);
    if (dx) {   /* the projection's share: dz W_in^T */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t r = 0; r < B * T; ++r)
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t j = 0; j < Z; ++j) acc += dz[r * Z + j] * W_in[p * Z + j];
                dx[r * P + p] += acc;
            }
    }
    return count;
}

/* dz at sampled rows, for sequences too long for sel_grad: the same window sums
 * mu_i = sum_{t=i}^{min(T-1,i+W-1)} gy_t C_t prod_{j=i+1..t} Abar_j and the same step and
 * output VJPs, evaluated at the sampled tokens only.  x [B,T,P] and target [B,T,P] are
 * the layer input and target, z [B,T,P+2N] its projection with the bias (any exact
 * evaluation of xhat W_in + [b_dt, 0, 0]).  The forward recurrence runs over every token
 * of each sampled sequence, keeping y only on the tokens some window needs.
 * samp_b[s], samp_t[s] (s < ns): the sampled rows; dz_out [ns, P+2N]. */
void sel_dz_rows(int64_t B, int64_t T, int64_t P, int64_t N, int64_t Tbar, const double *x, const double *A,
                 const double *z, const double *target, int64_t ns, const int64_t *samp_b, const int64_t *samp_t,
                 double *dz_out)
{
    const int64_t Z = P + 2 * N, PN = P * N, W = window_of(T, Tbar);
    (void)B;
    for (int64_t s = 0; s < ns; ++s) {
        const int64_t b = samp_b[s], i = samp_t[s];
        const int64_t tend = (i + W - 1 < T - 1) ? i + W - 1 : T - 1;
        const int64_t nw = tend - i + 1;
        double *gw = malloc(sizeof(double) * (size_t)(nw * P));    /* gy_t, t in [i, tend] */
        double *hp = calloc((size_t)PN, sizeof(double));           /* h_{i-1} */
        double *hi = malloc(sizeof(double) * (size_t)PN);          /* h_i */
        /* forward over [0, tend], channels in parallel */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t p = 0; p < P; ++p) {
            double *hv = calloc((size_t)N, sizeof(double));
            for (int64_t t = 0; t <= tend; ++t) {
                const int64_t r = b * T + t;
                const double *zr = z + r * Z;
                const double dt = softplus(zr[p]);
                double out = x[r * P + p];
                for (int64_t n = 0; n < N; ++n) {
                    hv[n] = exp(dt * A[p * N + n]) * hv[n] + dt * zr[P + n] * x[r * P + p];
                    out += zr[P + N + n] * hv[n];
                }
                if (t == i - 1)
                    for (int64_t n = 0; n < N; ++n) hp[p * N + n] = hv[n];
                if (t == i)
                    for (int64_t n = 0; n < N; ++n) hi[p * N + n] = hv[n];
                if (t >= i) gw[(t - i) * P + p] = out - target[r * P + p];
            }
            free(hv);
        }
        /* mu_i by its definition, then the VJPs of token i */
        double *mu = calloc((size_t)PN, sizeof(double));
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n) {
                double prod = 1.0, acc = 0.0;
                for (int64_t t = i; t <= tend; ++t) {
                    if (t > i) prod *= exp(softplus(z[(b * T + t) * Z + p]) * A[p * N + n]);
                    acc += gw[(t - i) * P + p] * z[(b * T + t) * Z + P + N + n] * prod;
                }
                mu[p * N + n] = acc;
            }
        const int64_t ri = b * T + i;
        const double *zr = z + ri * Z, *xr = x + ri * P;
        double *out = dz_out + s * Z;
        memset(out, 0, sizeof(double) * (size_t)Z);
        for (int64_t p = 0; p < P; ++p) {
            const double dt = softplus(zr[p]);
            double ddt = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double ab = exp(dt * A[p * N + n]);
                const double v = mu[p * N + n];
                ddt += v * (A[p * N + n] * ab * hp[p * N + n] + zr[P + n] * xr[p]);
                out[P + n] += v * dt * xr[p];
                out[P + N + n] += gw[p] * hi[p * N + n];
            }
            out[p] = ddt * sigmoid(zr[p]);
        }
        free(mu); free(gw); free(hp); free(hi);
    }
}
