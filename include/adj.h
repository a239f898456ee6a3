/*
 * adj.h -- C ABI of libadj.so, the GB300 (sm_103a) adjoint-sharding gradient path
 * for residual stacks of diagonal selective state-space layers.
 *
 * Source of the operations: the review page "Adjoint sharding for very long
 * context training of state space models" (pith.science), cited as [AS].
 *
 * Layer model ([AS] Assumptions: Sec. 3.1 SSM dynamics h_t = A_t h_{t-1} + B_t x_t,
 * y_t = C_t h_t; Sec. 3.2 residual structure y^K = y^0 + sum_k ytilde^k), in the
 * diagonal selective form A_t = diag(a_t), B_t xhat_t = u_t, C_t = W_o^T diag(c_t):
 *     a_t = sigmoid(xhat_t W_a + b_a),  u_t = xhat_t W_B,  c_t = xhat_t W_c,
 *     h_t = a_t . h_{t-1} + u_t  (h_0 = 0),   y_t = xhat_t + (c_t . h_t) W_o.
 *
 * Conventions shared by every call:
 *  - Arrays are row-major and token-major: [B,T,P] and [B,T,N] with the last
 *    index contiguous.  Every array pointer is a DEVICE pointer owned by the
 *    caller; the library never allocates, frees or keeps a pointer after a call.
 *  - Every pointer must be 16-byte aligned; P and N must be multiples of 8;
 *    B, T >= 0 are arbitrary (B*T == 0 launches nothing and returns ADJ_OK).
 *  - `ws` is caller-owned device scratch of at least adj_workspace_bytes() bytes,
 *    256-byte aligned.  Its first 256 bytes hold the sticky device status word
 *    read by adj_stream_status(); zero them once (cudaMemset) before first use.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on that stream.  Calls sharing one `ws` must be
 *    ordered on one stream.  A call enqueues only kernels and memsets on the
 *    stream (no allocation, no host synchronisation), so a sequence of calls can
 *    be captured into a CUDA graph and replayed; the graph keeps the pointers
 *    and sizes it was captured with.
 *  - Every argument is validated on the host before anything is launched; on an
 *    error nothing is launched and nothing is written.  Launch failures return
 *    ADJ_ECUDA.  Bounded device-side waits that give up record ADJ_ETIMEOUT in
 *    the workspace status word and return without hanging; read it with
 *    adj_stream_status().  Nothing throws, traps or exits.
 */
#ifndef ADJ_H_
#define ADJ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ADJ_OK = 0,
    ADJ_EINVAL = 1,      /* null pointer, bad enum, bad window */
    ADJ_ESHAPE = 2,      /* negative or unsupported sizes */
    ADJ_EALIGN = 3,      /* a pointer not 16-byte aligned (ws: 256-byte) */
    ADJ_EDTYPE = 4,      /* unsupported dtype combination */
    ADJ_EWORKSPACE = 5,  /* ws_bytes below adj_workspace_bytes() */
    ADJ_ECUDA = 6,       /* a CUDA launch or runtime call failed */
    ADJ_ETIMEOUT = 7     /* a bounded device wait gave up (see adj_stream_status) */
} adj_status;

typedef enum { ADJ_F32 = 0, ADJ_BF16 = 1 } adj_dtype;

/* Problem sizes and storage types of one layer call.
 * x_dtype: storage of the GEMM operands xhat, W_in, W_o (and of y_x below).
 * d_dtype: storage of the VJP factors D_a, D_u, D_c and of E. */
typedef struct {
    int64_t B, T;
    int32_t P, N;
    int32_t x_dtype, d_dtype;
} adj_dims;

/* Layer weights (device pointers).
 * W_in [P,3N] x_dtype: column blocks [W_a | W_B | W_c].
 * b_a  [N]   fp32.
 * W_o  [N,P] x_dtype. */
typedef struct {
    const void *W_in;
    const float *b_a;
    const void *W_o;
} adj_weights;

enum {
    ADJ_OP_FWD = 0, ADJ_OP_BWD_FULL = 1, ADJ_OP_BWD_TRUNC = 2, ADJ_OP_PARAM = 3, ADJ_OP_LOSS = 4,
    ADJ_OP_SEL_FWD = 5, ADJ_OP_SEL_BWD = 6, ADJ_OP_SEL_PARAM = 7   /* the general selective layer (below) */
};

/* Workspace bytes that call `op` needs for these sizes (Tbar: the window of
 * ADJ_OP_BWD_TRUNC and ADJ_OP_SEL_BWD, ignored otherwise).  One workspace of the maximum over the
 * ops used serves them all.  Returns 0 for invalid sizes. */
size_t adj_workspace_bytes(const adj_dims *dims, int op, int64_t Tbar);

/* Forward pass of one layer storing the states the adjoint needs
 * ([AS] Referee Report, comment on Algorithm 1: per-token, per-layer states are
 * kept; here a_t, c_t and h_t, the layer input being the caller's xhat).
 *   xhat [B,T,P] x_dtype  layer input as GEMM operand
 *   xres [B,T,P] fp32     residual input; NULL = use xhat's values
 *   a, c, h [B,T,N] fp32  stored gate, output gate and state (written)
 *   y    [B,T,P] fp32     layer output xres + (c . h) W_o (written; NULL to skip)
 *   y_x  [B,T,P] x_dtype  y rounded to x_dtype for the next layer's xhat
 *                         (written; NULL to skip; must be NULL if x_dtype is fp32) */
adj_status adj_fwd_scan(const adj_dims *dims, const adj_weights *w, const void *xhat,
                        const float *xres, float *a, float *c, float *h, float *y, void *y_x,
                        void *ws, size_t ws_bytes, void *stream);

/* Loss of the last layer and its cotangent: L = sum_{b,t} 1/2 ||y_t - target_t||^2,
 * gy = y - target.  y, target, gy [B,T,P] fp32 (gy written; may alias y);
 * gy_x [B,T,P] bf16: gy rounded to bf16 (written; NULL to skip; needs gy), the operand the
 * bf16 layers' backward GEMMs read (see gy_x of adj_bwd_* and adj_param_grad);
 * loss: one device double (written; NULL to skip).  Uses dims->B, T, P only. */
adj_status adj_loss_mse(const adj_dims *dims, const float *y, const float *target, float *gy,
                        void *gy_x, double *loss, void *ws, size_t ws_bytes, void *stream);

/* Adjoint pass of one layer, full window ([AS] Core claim, Proposition 2, with
 * lambda_{t,i} = C_t prod_{j=i+1..t} A_j; the sum over t of dl_t/dy_t lambda_{t,i}
 * is the reverse recurrence of [AS] What carries the argument, Proposition 1).
 * With g_t = gy_t W_o^T and mu_i = sum_{t>=i} g_t . c_t . prod_{j=i+1..t} a_j it
 * writes the per-token VJP seeds
 *   D_a = mu_i . h_{i-1} . a_i (1 - a_i)   (vjp^{A_i}),   D_u = mu_i   (vjp^{B_i}),
 *   D_c = g_t . h_t,  E = c_t . h_t        (vjp^{C_t}),
 * all [B,T,N] in d_dtype.  a, c, h [B,T,N] fp32 from adj_fwd_scan; gy [B,T,P]
 * fp32 = dL/dy of this layer (the total cotangent).  gy_x [B,T,P] bf16 (NULL to skip;
 * bf16 layers only): gy rounded to bf16, read in place of gy by the product g = gy W_o^T
 * (which rounds gy to bf16 in bf16 layers anyway).
 * dz [B*T, ceil(N/128)] fp32 (NULL to skip; needs w->b_a): per token and group of 128
 * channels, the sum of D_a z_a + D_u u + D_c c over the group, with the seeds as stored,
 * z_a = logit(a_t) - b_a = xhat_t W_a and u_t = h_t - a_t h_{t-1} = xhat_t W_B.  Summed
 * over the groups this is D_t . (xhat_t W_in) = xhat_t . dxhat_t, the row dot product
 * that adj_param_grad needs for a normalised layer input (see r and dz there). */
adj_status adj_bwd_full(const adj_dims *dims, const adj_weights *w, const float *a,
                        const float *c, const float *h, const float *gy, const void *gy_x, void *D_a,
                        void *D_u, void *D_c, void *E, float *dz, void *ws, size_t ws_bytes, void *stream);

/* As adj_bwd_full, truncated to the window Tbar ([AS] Core claim, last sentence;
 * Referee Report on Section 4.3): mu_i sums only t with t - i < Tbar.  Tbar >= 1;
 * Tbar >= T gives the full result. */
adj_status adj_bwd_trunc(const adj_dims *dims, const adj_weights *w, const float *a,
                         const float *c, const float *h, const float *gy, const void *gy_x, void *D_a,
                         void *D_u, void *D_c, void *E, float *dz, int64_t Tbar, void *ws, size_t ws_bytes,
                         void *stream);

/* Parameter gradients as reductions over all tokens ([AS] Core claim: the sum over
 * t and i of the VJPs, applied once per token to the summed seeds):
 *   dW_in [P,3N] = xhat^T [D_a | D_u | D_c],  db_a [N] = sum_t D_a,
 *   dW_o  [N,P]  = E^T gy,
 * fp32, overwritten (accumulate = 0) or added to (accumulate = 1).
 * The cotangent of the layer input, at most one of (NULL to skip):
 *   gy_prev [B,T,P] fp32 = gy + [D_a | D_u | D_c] W_in^T: the total cotangent of the
 *           layer below when that layer's output is this layer's input unchanged
 *           ([AS] residual identity; Proposition 3);
 *           with r and dz (both or neither): the layer input is the normalised residual
 *           stream xhat = y / r of adj_rms_norm, and gy_prev = gy + (dxhat - xhat m / P) / r
 *           with dxhat = [D_a | D_u | D_c] W_in^T and m = sum of dz's groups, the
 *           cotangent of y through the normalisation ([AS] Load-bearing premise); r [B,T]
 *           fp32 from adj_rms_norm, dz from adj_bwd_*, xhat as passed above;
 *   dxhat   [B,T,P] fp32 = [D_a | D_u | D_c] W_in^T alone (for adj_rms_norm_bwd).
 * bf16 layers only (NULL to skip): gy_x [B,T,P] bf16, gy rounded to bf16, read in place of
 * gy by the dW_o product; gy_prev_x [B,T,P] bf16, gy_prev rounded to bf16 (written; needs
 * gy_prev), the next layer's gy_x. */
adj_status adj_param_grad(const adj_dims *dims, const adj_weights *w, const void *xhat,
                          const void *D_a, const void *D_u, const void *D_c, const void *E,
                          const float *gy, const void *gy_x, float *dW_in, float *db_a, float *dW_o,
                          float *gy_prev, void *gy_prev_x, float *dxhat, const float *r, const float *dz,
                          int accumulate, void *ws, size_t ws_bytes, void *stream);

/* Normalised layer input of a stacked layer ([AS] Load-bearing premise: the layers
 * read "normalized inputs"): per token, xhat = y / r with
 * r = sqrt(mean_p y_p^2 + ADJ_NORM_EPS).  y [B,T,P] fp32 (the residual stream y^{k-1});
 * xhat [B,T,P] in dims->x_dtype and r [B,T] fp32 are written.  No workspace. */
#define ADJ_NORM_EPS 1e-6f
adj_status adj_rms_norm(const adj_dims *dims, const float *y, void *xhat, float *r, void *stream);

/* Cotangent through the normalisation: gy_prev = gy + (dxhat - xhat mean_p(xhat dxhat)) / r,
 * xhat = y / r recomputed from y [B,T,P] fp32 and r [B,T] from adj_rms_norm.
 * gy_prev [B,T,P] fp32 may alias dxhat or gy. */
adj_status adj_rms_norm_bwd(const adj_dims *dims, const float *y, const float *r, const float *dxhat,
                            const float *gy, float *gy_prev, void *stream);

/* ---------------------------------------------------------------------------
 * The general selective layer.  The pages give the layer only in its general form
 * h_t = A_t h_{t-1} + B_t xhat_t, y_t = C_t h_t with A_t, B_t, C_t functions of the token
 * ([AS] Circularity Check, assumptions); these calls take its selective reading, per
 * channel p < P and state n < N (N = 8 or 16):
 *     z_t = xhat_t W_in                      W_in [P, P+2N] = [W_dt | W_B | W_C]
 *     dt_t,p = softplus(z_t,p + b_dt,p),  B_t,n = z_t,P+n,  C_t,n = z_t,P+N+n
 *     Abar_t,pn = exp(dt_t,p A_pn)            A [P,N], the continuous-time decay
 *     h_t,pn = Abar_t,pn h_t-1,pn + dt_t,p B_t,n xhat_t,p   (h_-1 = 0)
 *     y_t,p = xres_t,p + sum_n C_t,n h_t,pn   (the residual identity; xres = xhat
 *                                             for a lone layer)
 * i.e. a PN-dimensional state with A_t = diag(Abar_t) and the full P x PN output map
 * C_t[p, (p,n)] = C_t,n.  Its gradient is the same sum over token pairs of independent
 * VJPs as the diagonal layer's ([AS] Core claim, Proposition 2), full or truncated to a
 * window.  Sizes: adj_dims with N = 8 or 16, P a multiple of 8, B <= 65535; x_dtype is
 * the storage of xhat and W_in, d_dtype that of dz.  h is [B,T,P,N] fp32 (state index
 * last).  No call waits on another CTA; adj_sel_bwd's waits for its own bulk copies are
 * bounded and record ADJ_ETIMEOUT in the workspace if one gives up.
 *
 * Stacks ([AS] What carries the argument: y^K = y^0 + sum_k ytilde^k; Load-bearing
 * premise: normalised inputs): layer 1 reads the input, layer k >= 2 reads the residual
 * stream y^{k-1} normalised per token, xhat^k = y^{k-1} / r (adj_rms_norm), with
 * xres = y^{k-1}.  Its input path then passes the cotangent down:
 *     gy^{k-1} = gy^k + (dxhat - xhat (xhat . dxhat) / P) / r,
 *     dxhat_t,p = (dz_t W_in^T)_p + dt_t,p sum_n mu_t,pn B_t,n
 * (the projection and the input term of the step), computed by adj_sel_bwd (r, gadd,
 * rowdot) and adj_sel_param_grad (gy_prev).
 * ------------------------------------------------------------------------- */
typedef struct {
    const void *W_in;    /* [P, P+2N] x_dtype */
    const float *b_dt;   /* [P] */
    const float *A;      /* [P, N] */
} adj_sel_weights;

/* Forward pass storing what the adjoint needs ([AS] Referee Report on Algorithm 1: the
 * per-token states are kept):
 *   xhat [B,T,P] x_dtype    layer input
 *   xres [B,T,P] fp32       residual input (NULL: xhat's values; a stacked layer passes
 *                           the residual stream y^{k-1} it normalised into xhat)
 *   z    [B,T,P+2N] fp32    xhat W_in, without b_dt (written)
 *   h    [B,T,P,N] fp32     states (written)
 *   y    [B,T,P] fp32       layer output (written; may not alias xres) */
adj_status adj_sel_fwd(const adj_dims *dims, const adj_sel_weights *w, const void *xhat, const float *xres,
                       float *z, float *h, float *y, void *ws, size_t ws_bytes, void *stream);

/* Columns of adj_sel_bwd's rowdot for these sizes (0 for sizes the selective calls reject). */
size_t adj_sel_rowdot_cols(const adj_dims *dims);

/* Adjoint of one selective layer for the cotangent gy = dL/dy [B,T,P] fp32: the window
 * sums mu_i = sum_{t=i}^{min(T-1, i+Tbar-1)} gy_t^T C_t prod_{j=i+1..t} A_j (all t >= i when
 * Tbar <= 0 or Tbar >= T; otherwise Tbar must be a multiple of 16), and the VJP of every
 * token's step and output map ([AS] Core claim, Proposition 2; last sentence: truncation):
 *   dz [B,T,P+2N] d_dtype   cotangent of z (written): columns p < P: the step's
 *                           (sum_n mu_pn (A_pn Abar_pn h_{t-1},pn + B_n xhat_p)) sigmoid(z_p + b_dt,p);
 *                           columns P+n: sum_p mu_pn dt_p xhat_p (B_t); P+N+n: sum_p gy_p h_t,pn (C_t)
 *   dA [P,N] fp32           sum_t mu_pn dt_p Abar_pn h_{t-1},pn (written)
 * xhat, z, h as written by adj_sel_fwd.
 * The input path of a stacked layer (all three or none; NULL for a lone layer or layer 1):
 *   r      [B,T] fp32                   the rms from adj_rms_norm (xhat = y^{k-1} / r)
 *   gadd   [B,T,P] fp32 (written)       gy + dt sum_n mu B / r, the input term's share
 *   rowdot [B*T, adj_sel_rowdot_cols] fp32 (written)  partial sums of xhat . dxhat, the
 *                                       projection's share taken as dz . z (z = xhat W_in,
 *                                       dz as stored), which adj_sel_param_grad sums
 * gadd may not alias gy. */
adj_status adj_sel_bwd(const adj_dims *dims, const adj_sel_weights *w, const void *xhat, const float *z,
                       const float *h, const float *gy, int64_t Tbar, void *dz, float *dA, const float *r,
                       float *gadd, float *rowdot, void *ws, size_t ws_bytes, void *stream);

/* Parameter gradients from dz ([AS] Core claim: the sum over tokens of the VJPs):
 *   dW_in [P, P+2N] fp32 = sum_t xhat_t^T dz_t,   db_dt [P] fp32 = sum_t dz_t[:P].
 * accumulate (0 or 1) adds into the outputs instead of overwriting them.
 * With the input path (r, gadd, rowdot from adj_sel_bwd and gy_prev, all or none; w->W_in
 * then required, w may be NULL otherwise): gy_prev [B,T,P] fp32 (written) =
 * gadd + (dz W_in^T - xhat m / P) / r with m the sum of rowdot's columns, the cotangent
 * of the residual stream y^{k-1} below. */
adj_status adj_sel_param_grad(const adj_dims *dims, const adj_sel_weights *w, const void *xhat, const void *dz,
                              float *dW_in, float *db_dt, const float *r, const float *gadd, const float *rowdot,
                              float *gy_prev, int accumulate, void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream`, return and clear the sticky device status of `ws`
 * (ADJ_OK or ADJ_ETIMEOUT); ADJ_ECUDA if the stream reports an error. */
adj_status adj_stream_status(void *ws, void *stream);

/* Static description of a status code. */
const char *adj_status_str(adj_status s);

/* The forward pass of adj_fwd_scan for callers that cannot allocate device memory
 * (the paper has no counterpart: it concerns how scratch memory is obtained).
 * Scratch comes from a 32 MiB array inside the library, which every GPU that loads
 * the library holds until the process exits, so no workspace is passed.  Inputs and
 * outputs are as in adj_fwd_scan.  Problems whose adj_workspace_bytes(dims,
 * ADJ_OP_FWD, 0) exceeds 32 MiB are rejected with ADJ_EWORKSPACE before anything is
 * launched.  `status` (device pointer to one unsigned, NULL to skip) receives the
 * call's device status word after the launches (non-zero: a bounded wait gave up).
 * The first call on a device looks up the array's device address and must come
 * before any stream capture.  All calls share the array: calls that overlap on the
 * GPU race.  Allocates nothing (no cudaMalloc/cudaFree). */
adj_status adj_fwd_scan_noalloc(const adj_dims *dims, const adj_weights *w, const void *xhat,
                                const float *xres, float *a, float *c, float *h, float *y, void *y_x,
                                unsigned *status, void *stream);

/* Failure-path self test (a library facility with no counterpart on the pages): runs
 * the bounded device waits the kernels rely on against objects that are never released.
 *   which & 1: the scans' decoupled look-back -- the forward state scan kernel runs over a
 *              small problem held in ws whose first chunk is never launched, so every
 *              other chunk waits for a predecessor that never publishes (a few seconds);
 *   which & 2: an mbarrier wait (TMA staging, GEMM pipeline) on a barrier that is never
 *              arrived on (about 2 s).
 * Each wait gives up after its limit, records the timeout in ws's status word and returns;
 * adj_stream_status(ws) then reports ADJ_ETIMEOUT.  ws: device memory, 256-byte aligned,
 * at least adj_selftest_ws_bytes() bytes, status word zero before the call. */
size_t adj_selftest_ws_bytes(void);
adj_status adj_selftest_waits(void *ws, size_t ws_bytes, int which, void *stream);

/* ---- Launch accounting and per-kernel timing (a library facility; the pages
 * describe no implementation, so these have no counterpart there).
 * adj_launch_count: kernels launched by this library since it was loaded.
 * adj_profile_enable(1): from now on every launch is bracketed by CUDA events
 *   on its stream; adj_profile_read(id, &n, &ms) synchronises on those events and
 *   returns the launch count and summed device time of kernel kind `id`
 *   (0 <= id < adj_profile_kernels(), named by adj_profile_name(id));
 *   adj_profile_reset() forgets all records.  Host-thread safe. */
unsigned long long adj_launch_count(void);
void adj_profile_enable(int on);
void adj_profile_reset(void);
int adj_profile_kernels(void);
const char *adj_profile_name(int id);
adj_status adj_profile_read(int id, int64_t *launches, double *total_ms);

#ifdef __cplusplus
}
#endif
#endif /* ADJ_H_ */
