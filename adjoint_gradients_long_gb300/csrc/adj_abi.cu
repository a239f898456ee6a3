// adj_abi.cu -- the extern "C" entry points of libadj.so: host-side validation,
// workspace layout and the launch sequence of each call.  The operations and their
// sources are documented in include/adj.h.
#include <string.h>

#include <algorithm>

#include "adj_internal.cuh"
#include "adj_profile.cuh"
#include "adj_sel.cuh"

using namespace adj;

namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// largest grid the scans launch (tickets are 32-bit)
constexpr int64_t MAX_CHUNKS = int64_t(1) << 31;

#define ADJ_TRY_(x)                                 \
    do {                                            \
        adj_status s_ = (x);                        \
        if (s_ != ADJ_OK) return s_;                \
    } while (0)

adj_status check_dims(const adj_dims *d) {
    if (!d) return ADJ_EINVAL;
    if (d->B < 0 || d->T < 0 || d->P <= 0 || d->N <= 0) return ADJ_ESHAPE;
    if (d->P % 8 || d->N % 8) return ADJ_ESHAPE;
    if ((d->x_dtype != ADJ_F32 && d->x_dtype != ADJ_BF16) || (d->d_dtype != ADJ_F32 && d->d_dtype != ADJ_BF16))
        return ADJ_EDTYPE;
    if (d->B * cdiv(d->N, 128) * cdiv(d->T, 32) >= MAX_CHUNKS) return ADJ_ESHAPE;
    return ADJ_OK;
}

// the general selective layer: N = 8 or 16 states a channel, one grid row per sequence
adj_status check_sel_dims(const adj_dims *d) {
    ADJ_TRY_(check_dims(d));
    if (d->N != 8 && d->N != 16) return ADJ_ESHAPE;
    if (d->B > 65535) return ADJ_ESHAPE;
    return ADJ_OK;
}

adj_status check_ptrs(std::initializer_list<const void *> ps) {
    for (const void *p : ps) {
        if (!p) return ADJ_EINVAL;
        if (!al16(p)) return ADJ_EALIGN;
    }
    return ADJ_OK;
}
adj_status check_opt(std::initializer_list<const void *> ps) {
    for (const void *p : ps)
        if (p && !al16(p)) return ADJ_EALIGN;
    return ADJ_OK;
}

// Largest split of the token reduction of a parameter-gradient GEMM: one wave of CTAs at
// 128 x 256 output tiles, at least 4 k-blocks of 64 tokens per split.  The launch lowers it
// when it takes narrower tiles, so that every CTA still owns one tile.
int gemm_splits(int64_t M, int64_t Nc, int64_t K) {
    const int64_t tiles = cdiv(M, 128) * cdiv(Nc, 256);
    int64_t s = 152 / tiles;
    if (s > K / 256) s = K / 256;
    if (s < 1) s = 1;
    if (s > 128) s = 128;
    return int(s);
}
int splits_in(const adj_dims *d) { return gemm_splits(d->P, 3 * int64_t(d->N), d->B * d->T); }
int splits_o(const adj_dims *d) { return gemm_splits(d->N, d->P, d->B * d->T); }
int colsum_blocks(const adj_dims *d) {
    int64_t n = cdiv(d->B * d->T, 64);   // four blocks on each of the 152 SMs for long inputs
    if (n > 608) n = 608;
    return n < 1 ? 1 : int(n);
}
int loss_blocks(int64_t count) {
    int64_t n = cdiv(count, 256 * 8);
    if (n > 608) n = 608;                 // four blocks on each of the 152 SMs
    return n < 1 ? 1 : int(n);
}

// Workspace layouts (offsets from ws; the first WS_HEADER bytes hold the status word).
struct Layout {
    size_t buf0 = 0, buf1 = 0, scan = 0, part0 = 0, part1 = 0, part2 = 0, wsplit = 0, total = 0;
};

Layout layout(const adj_dims *d, int op, int64_t Tbar) {
    Layout L;
    const size_t btn = al256(size_t(d->B * d->T) * d->N * 4);
    // fp32 weights are split once per call into bf16 hi/lo copies (4 bytes per value):
    // W_in and W_o for the forward, W_o for the backward, W_in for the input gradient
    const bool wsplit = d->x_dtype == ADJ_F32;
    const size_t win_s = wsplit ? al256(size_t(d->P) * 3 * d->N * 4) : 0;
    const size_t wo_s = wsplit ? al256(size_t(d->N) * d->P * 4) : 0;
    // the forward's W_in copy (interleaved columns; hi/lo for fp32 weights) is made for bf16
    // weights too
    const size_t win_f = al256(size_t(d->P) * 3 * d->N * (wsplit ? 4 : 2));
    size_t off = WS_HEADER;
    switch (op) {
    case ADJ_OP_FWD:            // u; bf16 layers: c . h in bf16 (the output projection's operand)
        L.buf0 = off; off += btn;
        if (d->x_dtype == ADJ_BF16) { L.buf1 = off; off += al256(size_t(d->B * d->T) * d->N * 2); }
        L.scan = off; off += scan_ws_bytes(d->B, d->T, d->N);
        L.wsplit = off; off += win_f + wo_s;
        break;
    case ADJ_OP_BWD_FULL:       // g
        L.buf0 = off; off += btn;
        L.scan = off; off += scan_ws_bytes(d->B, d->T, d->N);
        L.wsplit = off; off += wo_s;
        break;
    case ADJ_OP_BWD_TRUNC:      // g, R
        L.buf0 = off; off += btn;
        L.buf1 = off; off += (Tbar < d->T ? btn : 0);
        L.scan = off; off += std::max(scan_ws_bytes(d->B, d->T, d->N), al256(trunc_ws_bytes(d->B, d->T, d->N)));
        L.wsplit = off; off += wo_s;
        break;
    case ADJ_OP_PARAM: {
        L.part0 = off; off += al256(size_t(splits_in(d)) * d->P * 3 * d->N * 4);
        L.part1 = off; off += al256(size_t(splits_o(d)) * d->N * d->P * 4);
        L.part2 = off; off += al256(size_t(std::max(colsum_blocks(d), 2 * splits_in(d))) * d->N * 4);
        L.wsplit = off; off += win_s;
        break;
    }
    case ADJ_OP_LOSS:
        L.part0 = off; off += al256(size_t(loss_blocks(d->B * d->T * d->P)) * 8);
        break;
    case ADJ_OP_SEL_FWD: {      // chunk aggregates (2); fp32 weights: W_in's bf16 hi/lo split
        const size_t agg = al256(size_t(d->B * cdiv(d->T, sel_chunk(d->T, 0))) * d->P * d->N * 4);
        L.buf0 = off; off += agg;
        L.buf1 = off; off += agg;
        L.wsplit = off; off += wsplit ? al256(size_t(d->P) * (d->P + 2 * d->N) * 4) : 0;
        break;
    }
    case ADJ_OP_SEL_BWD: {      // aggregates (2, 4 truncated), R (truncated), dB/dC and dA partials
        const bool tr = Tbar > 0 && Tbar < d->T;
        const int64_t nch = cdiv(d->T, sel_chunk(d->T, tr ? Tbar : 0));
        const size_t agg = al256(size_t(d->B * nch) * d->P * d->N * 4);
        L.buf0 = off; off += (tr ? 4 : 2) * agg;
        L.buf1 = off; off += tr ? al256(size_t(d->B * d->T) * d->P * d->N * 4) : 0;
        L.part0 = off; off += al256(size_t(d->B * d->T) * sel_slices(d->P, d->N) * 2 * d->N * 4);
        L.part1 = off; off += agg;
        break;
    }
    case ADJ_OP_SEL_PARAM: {    // dW_in split partials, db_dt block partials; fp32: W_in's split
        const int64_t zw = d->P + 2 * int64_t(d->N);
        L.part0 = off; off += al256(size_t(gemm_splits(d->P, zw, d->B * d->T)) * d->P * zw * 4);
        L.part1 = off; off += al256(size_t(colsum_blocks(d)) * d->P * 4);
        L.wsplit = off; off += wsplit ? al256(size_t(d->P) * zw * 4) : 0;
        break;
    }
    default:
        return Layout{};
    }
    L.total = off;
    return L;
}

adj_status check_ws(const adj_dims *d, int op, int64_t Tbar, void *ws, size_t ws_bytes, Layout *L) {
    *L = layout(d, op, Tbar);
    if (!ws) return ADJ_EINVAL;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return ADJ_EALIGN;
    if (ws_bytes < L->total) return ADJ_EWORKSPACE;
    return ADJ_OK;
}

inline char *at(void *ws, size_t off) { return static_cast<char *>(ws) + off; }
inline unsigned *status_word(void *ws) { return static_cast<unsigned *>(ws); }

#define ADJ_TRY(x)                                  \
    do {                                            \
        adj_status s_ = (x);                        \
        if (s_ != ADJ_OK) return s_;                \
    } while (0)
#define ADJ_CUDA(x)                                 \
    do {                                            \
        if ((x) != cudaSuccess) return ADJ_ECUDA;   \
    } while (0)

GemmOperand op1(const void *p, int64_t s_row, int64_t s_k, bool bf16, const float *mul = nullptr) {
    GemmOperand o;
    o.p[0] = p; o.p[1] = p; o.p[2] = p;
    o.lo[0] = o.lo[1] = o.lo[2] = nullptr;
    o.blk = int64_t(1) << 62;
    o.s_row = s_row; o.s_k = s_k; o.bf16 = bf16; o.mul = mul;
    return o;
}
GemmOperand op3(const void *p0, const void *p1, const void *p2, int64_t blk, int64_t s_row, int64_t s_k, bool bf16) {
    GemmOperand o;
    o.p[0] = p0; o.p[1] = p1; o.p[2] = p2;
    o.lo[0] = o.lo[1] = o.lo[2] = nullptr;
    o.blk = blk; o.s_row = s_row; o.s_k = s_k; o.bf16 = bf16; o.mul = nullptr;
    return o;
}
// A weight operand: fp32 weights are split into bf16 hi/lo copies at `split` (n values
// each) for the split-precision GEMM; bf16 weights are used as they are.
GemmOperand opw(const void *w, int64_t n, bool xbf, void *split, int64_t s_row, int64_t s_k, cudaStream_t st,
                cudaError_t *err) {
    if (xbf) return op1(w, s_row, s_k, true);
    __nv_bfloat16 *hi = static_cast<__nv_bfloat16 *>(split), *lo = hi + n;
    ProfScope ps(K_WEIGHT_PREP, st);
    *err = launch_split_bf16(static_cast<const float *>(w), n, hi, lo, st);
    GemmOperand o = op1(hi, s_row, s_k, true);
    o.lo[0] = o.lo[1] = o.lo[2] = lo;
    return o;
}
GemmEpilogue epi(Epi k) {
    GemmEpilogue e;
    memset(&e, 0, sizeof(e));
    e.kind = k;
    return e;
}

adj_status bwd_common(const adj_dims *dims, const adj_weights *w, const float *a, const float *c, const float *h,
                      const float *gy, const void *gy_x, void *D_a, void *D_u, void *D_c, void *E, float *dz,
                      int64_t Tbar, int op, void *ws, size_t ws_bytes, void *stream) {
    ADJ_TRY(check_dims(dims));
    if (!w) return ADJ_EINVAL;
    ADJ_TRY(check_ptrs({w->W_o, a, c, h, gy, D_a, D_u, D_c, E}));
    ADJ_TRY(check_opt({dz, gy_x}));
    if (gy_x && dims->x_dtype != ADJ_BF16) return ADJ_EINVAL;
    if (dz) ADJ_TRY(check_ptrs({w->b_a}));
    if (op == ADJ_OP_BWD_TRUNC && Tbar < 1) return ADJ_EINVAL;
    Layout L;
    ADJ_TRY(check_ws(dims, op, Tbar, ws, ws_bytes, &L));
    const int64_t B = dims->B, T = dims->T, BT = B * T;
    const int P = dims->P, N = dims->N;
    if (BT == 0) return ADJ_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *g = reinterpret_cast<float *>(at(ws, L.buf0));
    // g = gy W_o^T  (the cotangent of c . h)
    GemmEpilogue e = epi(Epi::Store);
    e.out0 = g;
    e.ld = N;
    {
        cudaError_t err = cudaSuccess;
        const GemmOperand Wo = opw(w->W_o, int64_t(N) * P, dims->x_dtype == ADJ_BF16, at(ws, L.wsplit), P, 1, st, &err);
        ADJ_CUDA(err);
        ProfScope ps(K_COT_PROJ, st);
        // bf16 layers with the cotangent's bf16 copy: the GEMM reads it by TMA (the same
        // rounding the fp32 operand would get in its conversion)
        const GemmOperand A = gy_x ? op1(gy_x, P, 1, true) : op1(gy, P, 1, false);
        ADJ_CUDA(launch_gemm_tc(BT, N, P, A, Wo, e, 1, dims->x_dtype == ADJ_F32, status_word(ws), st));
    }
    const bool trunc = op == ADJ_OP_BWD_TRUNC && Tbar < T;
    float *R = nullptr;
    if (trunc && trunc_one_launch(T, Tbar)) {
        // windows of whole scan chunks: the window scan and the reverse scan in one launch
        ProfScope ps(K_BWD_SCAN, st);
        ADJ_CUDA(launch_trunc_scan(g, c, a, h, reinterpret_cast<float *>(at(ws, L.buf1)), D_a, D_u, D_c, E,
                                   dims->d_dtype == ADJ_BF16, B, T, N, Tbar, at(ws, L.scan), status_word(ws), st,
                                   dz ? w->b_a : nullptr, dz));
        return ADJ_OK;
    }
    if (trunc) {
        R = reinterpret_cast<float *>(at(ws, L.buf1));
        ProfScope ps(K_WIN_SCAN, st);
        ADJ_CUDA(launch_win_scan(g, c, a, R, B, T, N, Tbar, at(ws, L.scan), status_word(ws), st));
    }
    ProfScope ps(K_BWD_SCAN, st);
    ADJ_CUDA(launch_bwd_scan(g, c, a, h, R, D_a, D_u, D_c, E, dims->d_dtype == ADJ_BF16, B, T, N, trunc ? Tbar : 0,
                             at(ws, L.scan), status_word(ws), st, dz ? w->b_a : nullptr, dz));
    return ADJ_OK;
}

}  // namespace

extern "C" {

size_t adj_workspace_bytes(const adj_dims *dims, int op, int64_t Tbar) {
    if (check_dims(dims) != ADJ_OK) return 0;
    if (op == ADJ_OP_BWD_TRUNC && Tbar < 1) return 0;
    if ((op == ADJ_OP_SEL_FWD || op == ADJ_OP_SEL_BWD || op == ADJ_OP_SEL_PARAM) && check_sel_dims(dims) != ADJ_OK)
        return 0;
    if (op == ADJ_OP_SEL_BWD && !sel_window_ok(dims->T, Tbar)) return 0;
    return layout(dims, op, Tbar).total;
}

adj_status adj_fwd_scan(const adj_dims *dims, const adj_weights *w, const void *xhat, const float *xres, float *a,
                        float *c, float *h, float *y, void *y_x, void *ws, size_t ws_bytes, void *stream) {
    ADJ_TRY(check_dims(dims));
    if (!w) return ADJ_EINVAL;
    ADJ_TRY(check_ptrs({w->W_in, w->b_a, w->W_o, xhat, a, c, h}));
    ADJ_TRY(check_opt({xres, y, y_x}));
    if (y_x && (!y || dims->x_dtype != ADJ_BF16)) return ADJ_EINVAL;
    Layout L;
    ADJ_TRY(check_ws(dims, ADJ_OP_FWD, 0, ws, ws_bytes, &L));
    const int64_t B = dims->B, T = dims->T, BT = B * T;
    const int P = dims->P, N = dims->N;
    if (BT == 0) return ADJ_OK;
    const bool xbf = dims->x_dtype == ADJ_BF16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *u = reinterpret_cast<float *>(at(ws, L.buf0));
    // [z_a | u | c] = xhat W_in;  a = sigmoid(z_a + b_a)
    GemmEpilogue e = epi(Epi::ProjIn);
    e.out0 = a; e.out1 = u; e.out2 = c; e.bias = w->b_a; e.N = N;
    cudaError_t err = cudaSuccess;
    GemmOperand Win;
    // W_o's bf16 hi/lo split (fp32 weights), made with W_in's copy when there is one
    __nv_bfloat16 *wo_hi = reinterpret_cast<__nv_bfloat16 *>(at(ws, L.wsplit + al256(size_t(P) * 3 * N * (xbf ? 2 : 4))));
    bool wo_done = false;
    if (N % 32 == 0) {
        // interleave the a, u, c column chunks so every output tile carries a share of the
        // sigmoid (the epilogue maps the chunks back)
        __nv_bfloat16 *hi = reinterpret_cast<__nv_bfloat16 *>(at(ws, L.wsplit));
        __nv_bfloat16 *lo = xbf ? nullptr : hi + int64_t(P) * 3 * N;
        wo_done = y && !xbf;
        {
            ProfScope pw(K_WEIGHT_PREP, st);
            ADJ_CUDA(launch_prep_win(w->W_in, xbf, P, N, hi, lo, st, wo_done ? static_cast<const float *>(w->W_o) : nullptr,
                                     wo_hi, wo_hi + int64_t(N) * P));
        }
        Win = op1(hi, 1, 3 * int64_t(N), true);
        if (lo) Win.lo[0] = Win.lo[1] = Win.lo[2] = lo;
        e.interleave = true;
    } else {
        Win = opw(w->W_in, int64_t(P) * 3 * N, xbf, at(ws, L.wsplit), 1, 3 * int64_t(N), st, &err);
        ADJ_CUDA(err);
    }
    {
        ProfScope ps(K_PROJ_IN, st);
        ADJ_CUDA(launch_gemm_tc(BT, 3 * int64_t(N), P, op1(xhat, P, 1, xbf), Win, e, 1, !xbf, status_word(ws), st));
    }
    // h_t = a_t h_{t-1} + u_t; bf16 layers that want y also get c . h rounded to bf16 (the
    // output projection's A operand, loaded by TMA straight into the MMA layout)
    __nv_bfloat16 *chx = (y && xbf) ? reinterpret_cast<__nv_bfloat16 *>(at(ws, L.buf1)) : nullptr;
    {
        ProfScope ps(K_FWD_SCAN, st);
        ADJ_CUDA(launch_fwd_scan(a, u, h, B, T, N, at(ws, L.scan), status_word(ws), st, false, chx ? c : nullptr, chx));
    }
    if (y) {
        // y = xres + (c . h) W_o
        GemmEpilogue e2 = epi(Epi::StoreAdd);
        e2.out0 = y; e2.out_x = y_x; e2.ld = P;
        e2.add = xres ? static_cast<const void *>(xres) : xhat;
        e2.add_bf16 = !xres && xbf;
        GemmOperand Wo;
        if (wo_done) {
            Wo = op1(wo_hi, 1, P, true);
            Wo.lo[0] = Wo.lo[1] = Wo.lo[2] = wo_hi + int64_t(N) * P;
        } else {
            Wo = opw(w->W_o, int64_t(N) * P, xbf, wo_hi, 1, P, st, &err);
            ADJ_CUDA(err);
        }
        ProfScope ps(K_PROJ_OUT, st);
        const GemmOperand A = chx ? op1(chx, N, 1, true) : op1(c, N, 1, false, h);
        ADJ_CUDA(launch_gemm_tc(BT, P, N, A, Wo, e2, 1, !xbf, status_word(ws), st));
    }
    return ADJ_OK;
}

adj_status adj_loss_mse(const adj_dims *dims, const float *y, const float *target, float *gy, void *gy_x,
                        double *loss, void *ws, size_t ws_bytes, void *stream) {
    ADJ_TRY(check_dims(dims));
    ADJ_TRY(check_ptrs({y, target}));
    ADJ_TRY(check_opt({gy, gy_x, loss}));
    if (!gy && !loss) return ADJ_EINVAL;
    if (gy_x && !gy) return ADJ_EINVAL;
    Layout L;
    ADJ_TRY(check_ws(dims, ADJ_OP_LOSS, 0, ws, ws_bytes, &L));
    const int64_t count = dims->B * dims->T * dims->P;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (count == 0) {
        if (loss) ADJ_CUDA(cudaMemsetAsync(loss, 0, sizeof(double), st));
        return ADJ_OK;
    }
    ProfScope ps(K_LOSS, st);
    ADJ_CUDA(launch_loss(y, target, gy, static_cast<__nv_bfloat16 *>(gy_x), count,
                         reinterpret_cast<double *>(at(ws, L.part0)), loss_blocks(count),
                         status_word(ws) + 1, loss, st));
    return ADJ_OK;
}

adj_status adj_bwd_full(const adj_dims *dims, const adj_weights *w, const float *a, const float *c, const float *h,
                        const float *gy, const void *gy_x, void *D_a, void *D_u, void *D_c, void *E, float *dz,
                        void *ws, size_t ws_bytes, void *stream) {
    return bwd_common(dims, w, a, c, h, gy, gy_x, D_a, D_u, D_c, E, dz, 0, ADJ_OP_BWD_FULL, ws, ws_bytes, stream);
}

adj_status adj_bwd_trunc(const adj_dims *dims, const adj_weights *w, const float *a, const float *c, const float *h,
                         const float *gy, const void *gy_x, void *D_a, void *D_u, void *D_c, void *E, float *dz,
                         int64_t Tbar, void *ws, size_t ws_bytes, void *stream) {
    return bwd_common(dims, w, a, c, h, gy, gy_x, D_a, D_u, D_c, E, dz, Tbar, ADJ_OP_BWD_TRUNC, ws, ws_bytes,
                      stream);
}

adj_status adj_param_grad(const adj_dims *dims, const adj_weights *w, const void *xhat, const void *D_a,
                          const void *D_u, const void *D_c, const void *E, const float *gy, const void *gy_x,
                          float *dW_in, float *db_a, float *dW_o, float *gy_prev, void *gy_prev_x, float *dxhat,
                          const float *r, const float *dz, int accumulate, void *ws, size_t ws_bytes, void *stream) {
    ADJ_TRY(check_dims(dims));
    if (!w) return ADJ_EINVAL;
    ADJ_TRY(check_ptrs({w->W_in, xhat, D_a, D_u, D_c, E, gy, dW_in, db_a, dW_o}));
    ADJ_TRY(check_opt({gy_x, gy_prev, gy_prev_x, dxhat, r, dz}));
    if (gy_prev && dxhat) return ADJ_EINVAL;
    if ((gy_x || gy_prev_x) && dims->x_dtype != ADJ_BF16) return ADJ_EINVAL;
    if (gy_prev_x && !gy_prev) return ADJ_EINVAL;
    if ((r != nullptr) != (dz != nullptr) || (r && !gy_prev)) return ADJ_EINVAL;
    if (accumulate != 0 && accumulate != 1) return ADJ_EINVAL;
    Layout L;
    ADJ_TRY(check_ws(dims, ADJ_OP_PARAM, 0, ws, ws_bytes, &L));
    const int64_t BT = dims->B * dims->T;
    const int P = dims->P, N = dims->N;
    const bool xbf = dims->x_dtype == ADJ_BF16, dbf = dims->d_dtype == ADJ_BF16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (BT == 0) {
        if (!accumulate) {
            ADJ_CUDA(cudaMemsetAsync(dW_in, 0, size_t(P) * 3 * N * 4, st));
            ADJ_CUDA(cudaMemsetAsync(db_a, 0, size_t(N) * 4, st));
            ADJ_CUDA(cudaMemsetAsync(dW_o, 0, size_t(N) * P * 4, st));
        }
        return ADJ_OK;
    }
    const int s_in = splits_in(dims), s_o = splits_o(dims);
    int su_in = s_in, su_o = s_o;   // split counts the launches took (at most the above)
    float *part_in = reinterpret_cast<float *>(at(ws, L.part0));
    float *part_o = reinterpret_cast<float *>(at(ws, L.part1));
    // dW_in = xhat^T [D_a | D_u | D_c]; with fp32 seeds the producers also sum D_a's
    // columns (db_a partials, two a split) while they convert the raw tiles
    float *part_c = reinterpret_cast<float *>(at(ws, L.part2));
    GemmEpilogue e = epi(Epi::Partial);
    e.out0 = part_in;
    e.csum = part_c;
    e.csum_n = N;
    bool csum_done = false;
    {
        ProfScope ps(K_PARAM_DWIN, st);
        ADJ_CUDA(launch_gemm_tc(P, 3 * int64_t(N), BT, op1(xhat, 1, P, xbf), op3(D_a, D_u, D_c, N, 1, N, dbf), e, s_in,
                                !xbf, status_word(ws), st, &su_in, &csum_done));
    }
    // otherwise db_a = sum_t D_a: block partials while D_a is still partly in L2
    int ncs = 2 * su_in;
    if (!csum_done) {
        ncs = colsum_blocks(dims);
        ProfScope ps(K_COLSUM, st);
        ADJ_CUDA(launch_colsum(D_a, dbf, BT, N, part_c, ncs, st));
    }
    // dW_o = E^T gy
    GemmEpilogue e2 = epi(Epi::Partial);
    e2.out0 = part_o;
    {
        ProfScope ps(K_PARAM_DWO, st);
        const GemmOperand Bg = gy_x ? op1(gy_x, 1, P, true) : op1(gy, 1, P, false);
        ADJ_CUDA(launch_gemm_tc(N, P, BT, op1(E, 1, N, dbf), Bg, e2, s_o, !xbf, status_word(ws), st, &su_o));
    }
    // the three sums over partials, in one launch
    {
        const RedSeg segs[3] = {{part_in, dW_in, int64_t(P) * 3 * N / 4, su_in, 0, 0},
                                {part_o, dW_o, int64_t(N) * P / 4, su_o, 0, 0},
                                {part_c, db_a, N / 4, ncs, 0, 0}};
        ProfScope ps(K_PARAM_REDUCE, st);
        ADJ_CUDA(launch_reduce_partials(segs, 3, accumulate, st));
    }
    if (gy_prev || dxhat) {
        // dxhat = [D_a | D_u | D_c] W_in^T, or gy_prev = gy + dxhat, or, through a normalised
        // input xhat = y / r, gy_prev = gy + (dxhat - xhat (xhat . dxhat) / P) / r with the row
        // dot products xhat . dxhat = sum of dz over the channel slices
        GemmEpilogue e3 = epi(gy_prev ? Epi::StoreAdd : Epi::Store);
        e3.out0 = gy_prev ? gy_prev : dxhat; e3.add = gy; e3.ld = P;
        e3.out_x = gy_prev_x;   // the bf16 copy of gy_prev for the next layer's GEMMs
        if (r) {
            e3.nr = r;
            e3.ndz = dz;
            e3.nsl = int(cdiv(N, 128));
            e3.nx = xhat;
            e3.nx_bf16 = xbf;
            e3.inv_P = 1.f / float(P);
        }
        cudaError_t err = cudaSuccess;
        const GemmOperand Win = opw(w->W_in, int64_t(P) * 3 * N, xbf, at(ws, L.wsplit), 3 * int64_t(N), 1, st, &err);
        ADJ_CUDA(err);
        ProfScope ps(K_INPUT_GRAD, st);
        ADJ_CUDA(launch_gemm_tc(BT, P, 3 * int64_t(N), op3(D_a, D_u, D_c, N, N, 1, dbf), Win, e3, 1, !xbf,
                                status_word(ws), st));
    }
    return ADJ_OK;
}

adj_status adj_rms_norm(const adj_dims *dims, const float *y, void *xhat, float *r, void *stream) {
    ADJ_TRY(check_dims(dims));
    ADJ_TRY(check_ptrs({y, xhat, r}));
    const int64_t rows = dims->B * dims->T;
    if (rows == 0) return ADJ_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ProfScope ps(K_RMS_NORM, st);
    ADJ_CUDA(launch_rms_norm(y, xhat, dims->x_dtype == ADJ_BF16, r, rows, dims->P, ADJ_NORM_EPS, st));
    return ADJ_OK;
}

adj_status adj_rms_norm_bwd(const adj_dims *dims, const float *y, const float *r, const float *dxhat,
                            const float *gy, float *gy_prev, void *stream) {
    ADJ_TRY(check_dims(dims));
    ADJ_TRY(check_ptrs({y, r, dxhat, gy, gy_prev}));
    const int64_t rows = dims->B * dims->T;
    if (rows == 0) return ADJ_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ProfScope ps(K_RMS_NORM_BWD, st);
    ADJ_CUDA(launch_rms_norm_bwd(y, r, dxhat, gy, gy_prev, rows, dims->P, st));
    return ADJ_OK;
}

// ---------------------------------------------------------------- the general selective layer
size_t adj_sel_rowdot_cols(const adj_dims *dims) {
    if (check_sel_dims(dims) != ADJ_OK) return 0;
    return size_t(sel_slices(dims->P, dims->N)) + 1;
}

adj_status adj_sel_fwd(const adj_dims *dims, const adj_sel_weights *w, const void *xhat, const float *xres, float *z,
                       float *h, float *y, void *ws, size_t ws_bytes, void *stream) {
    ADJ_TRY(check_sel_dims(dims));
    if (!w) return ADJ_EINVAL;
    ADJ_TRY(check_ptrs({w->W_in, w->b_dt, w->A, xhat, z, h, y}));
    ADJ_TRY(check_opt({xres}));
    Layout L;
    ADJ_TRY(check_ws(dims, ADJ_OP_SEL_FWD, 0, ws, ws_bytes, &L));
    const int64_t B = dims->B, T = dims->T, BT = B * T;
    const int P = dims->P, N = dims->N;
    if (BT == 0) return ADJ_OK;
    const bool xbf = dims->x_dtype == ADJ_BF16;
    const int64_t zw = P + 2 * int64_t(N);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // z = xhat W_in
    {
        cudaError_t err = cudaSuccess;
        const GemmOperand Win = opw(w->W_in, int64_t(P) * zw, xbf, at(ws, L.wsplit), 1, zw, st, &err);
        ADJ_CUDA(err);
        GemmEpilogue e = epi(Epi::Store);
        e.out0 = z;
        e.ld = zw;
        ProfScope ps(K_SEL_PROJ, st);
        ADJ_CUDA(launch_gemm_tc(BT, zw, P, op1(xhat, P, 1, xbf), Win, e, 1, !xbf, status_word(ws), st));
    }
    ProfScope ps(K_SEL_FWD, st, 3);
    ADJ_CUDA(launch_sel_fwd(z, xhat, xbf, w->b_dt, w->A, h, y, xres, reinterpret_cast<float *>(at(ws, L.buf0)),
                            reinterpret_cast<float *>(at(ws, L.buf1)), B, T, P, N, st));
    return ADJ_OK;
}

adj_status adj_sel_bwd(const adj_dims *dims, const adj_sel_weights *w, const void *xhat, const float *z,
                       const float *h, const float *gy, int64_t Tbar, void *dz, float *dA, const float *r, float *gadd,
                       float *rowdot, void *ws, size_t ws_bytes, void *stream) {
    ADJ_TRY(check_sel_dims(dims));
    if (!w) return ADJ_EINVAL;
    ADJ_TRY(check_ptrs({w->b_dt, w->A, xhat, z, h, gy, dz, dA}));
    ADJ_TRY(check_opt({r, gadd, rowdot}));
    if ((r != nullptr) != (gadd != nullptr) || (r != nullptr) != (rowdot != nullptr)) return ADJ_EINVAL;
    if (!sel_window_ok(dims->T, Tbar)) return ADJ_EINVAL;
    Layout L;
    ADJ_TRY(check_ws(dims, ADJ_OP_SEL_BWD, Tbar, ws, ws_bytes, &L));
    const int64_t B = dims->B, T = dims->T, BT = B * T;
    const int P = dims->P, N = dims->N;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (BT == 0) {
        ADJ_CUDA(cudaMemsetAsync(dA, 0, size_t(P) * N * 4, st));
        return ADJ_OK;
    }
    const bool tr = Tbar > 0 && Tbar < T;
    const size_t agg = al256(size_t(B * cdiv(T, sel_chunk(T, tr ? Tbar : 0))) * P * N * 4);
    SelBwdWs sw;
    sw.aggX = reinterpret_cast<float *>(at(ws, L.buf0));
    sw.aggY = reinterpret_cast<float *>(at(ws, L.buf0 + agg));
    sw.winX = tr ? reinterpret_cast<float *>(at(ws, L.buf0 + 2 * agg)) : nullptr;
    sw.winY = tr ? reinterpret_cast<float *>(at(ws, L.buf0 + 3 * agg)) : nullptr;
    sw.R = tr ? reinterpret_cast<float *>(at(ws, L.buf1)) : nullptr;
    sw.bc = reinterpret_cast<float *>(at(ws, L.part0));
    sw.dAp = reinterpret_cast<float *>(at(ws, L.part1));
    ProfScope ps(K_SEL_BWD, st, tr ? 7 : 5);
    SelInp inp;
    inp.r = r;
    inp.gadd = gadd;
    inp.rowdot = rowdot;
    ADJ_CUDA(launch_sel_bwd(z, xhat, dims->x_dtype == ADJ_BF16, gy, h, w->b_dt, w->A, dz, dims->d_dtype == ADJ_BF16, dA,
                            sw, inp, B, T, P, N, tr ? Tbar : 0, status_word(ws), st));
    return ADJ_OK;
}

adj_status adj_sel_param_grad(const adj_dims *dims, const adj_sel_weights *w, const void *xhat, const void *dz,
                              float *dW_in, float *db_dt, const float *r, const float *gadd, const float *rowdot,
                              float *gy_prev, int accumulate, void *ws, size_t ws_bytes, void *stream) {
    ADJ_TRY(check_sel_dims(dims));
    ADJ_TRY(check_ptrs({xhat, dz, dW_in, db_dt}));
    ADJ_TRY(check_opt({r, gadd, rowdot, gy_prev}));
    const bool inpath = gy_prev != nullptr;
    if ((r != nullptr) != inpath || (gadd != nullptr) != inpath || (rowdot != nullptr) != inpath) return ADJ_EINVAL;
    if (inpath && (!w || !w->W_in)) return ADJ_EINVAL;
    if (inpath) ADJ_TRY(check_ptrs({w->W_in}));
    if (accumulate != 0 && accumulate != 1) return ADJ_EINVAL;
    Layout L;
    ADJ_TRY(check_ws(dims, ADJ_OP_SEL_PARAM, 0, ws, ws_bytes, &L));
    const int64_t BT = dims->B * dims->T;
    const int P = dims->P, N = dims->N;
    const int64_t zw = P + 2 * int64_t(N);
    const bool xbf = dims->x_dtype == ADJ_BF16, dbf = dims->d_dtype == ADJ_BF16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (BT == 0) {
        if (!accumulate) {
            ADJ_CUDA(cudaMemsetAsync(dW_in, 0, size_t(P) * zw * 4, st));
            ADJ_CUDA(cudaMemsetAsync(db_dt, 0, size_t(P) * 4, st));
        }
        return ADJ_OK;
    }
    const int s = gemm_splits(P, zw, BT);
    int su = s;
    float *part = reinterpret_cast<float *>(at(ws, L.part0));
    float *part_b = reinterpret_cast<float *>(at(ws, L.part1));
    GemmEpilogue e = epi(Epi::Partial);
    e.out0 = part;
    {
        ProfScope ps(K_SEL_DW, st);
        ADJ_CUDA(launch_gemm_tc(P, zw, BT, op1(xhat, 1, P, xbf), op1(dz, 1, zw, dbf), e, s, !xbf, status_word(ws), st,
                                &su));
    }
    const int nb = colsum_blocks(dims);
    {
        ProfScope ps(K_COLSUM, st);
        ADJ_CUDA(launch_sel_colsum(dz, dbf, BT, P, int(zw), nb, part_b, st));
    }
    const RedSeg segs[2] = {{part, dW_in, int64_t(P) * zw / 4, su, 0, 0}, {part_b, db_dt, P / 4, nb, 0, 0}};
    {
        ProfScope ps(K_PARAM_REDUCE, st);
        ADJ_CUDA(launch_reduce_partials(segs, 2, accumulate, st));
    }
    if (inpath) {
        // the cotangent of the residual stream below: with dxhat = dz W_in^T + dxd,
        // gy_prev = gy + (dxhat - xhat (xhat . dxhat) / P) / r, where gadd = gy + dxd / r
        // and the row dots xhat . dxhat come summed over rowdot's slices
        GemmEpilogue e3 = epi(Epi::StoreAdd);
        e3.out0 = gy_prev;
        e3.add = gadd;
        e3.ld = P;
        e3.nr = r;
        e3.ndz = rowdot;
        e3.nsl = sel_slices(P, N) + 1;
        e3.nx = xhat;
        e3.nx_bf16 = xbf;
        e3.inv_P = 1.f / float(P);
        cudaError_t err = cudaSuccess;
        const GemmOperand Win = opw(w->W_in, int64_t(P) * zw, xbf, at(ws, L.wsplit), zw, 1, st, &err);
        ADJ_CUDA(err);
        ProfScope ps(K_SEL_DX, st);
        ADJ_CUDA(launch_gemm_tc(BT, P, zw, op1(dz, zw, 1, dbf), Win, e3, 1, !xbf, status_word(ws), st));
    }
    return ADJ_OK;
}

adj_status adj_stream_status(void *ws, void *stream) {
    if (!ws) return ADJ_EINVAL;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return ADJ_EALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return ADJ_ECUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return ADJ_ECUDA;
    if (word) {
        if (cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return ADJ_ECUDA;
        return ADJ_ETIMEOUT;
    }
    return ADJ_OK;
}

const char *adj_status_str(adj_status s) {
    switch (s) {
    case ADJ_OK: return "ok";
    case ADJ_EINVAL: return "invalid argument";
    case ADJ_ESHAPE: return "unsupported shape";
    case ADJ_EALIGN: return "misaligned pointer";
    case ADJ_EDTYPE: return "unsupported dtype";
    case ADJ_EWORKSPACE: return "workspace too small";
    case ADJ_ECUDA: return "CUDA error";
    case ADJ_ETIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
