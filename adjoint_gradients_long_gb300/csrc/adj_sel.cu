// adj_sel.cu -- the general selective layer's scans: forward state scan, window scan and
// reverse adjoint scan with the fused per-token VJP formation.
//
// Source: the review page "Adjoint sharding for very long context training of state
// space models" ([AS]).  The layer is the pages' general form h_t = A_t h_{t-1} + B_t xhat_t,
// y_t = C_t h_t ([AS] Circularity Check, assumptions) in its selective reading, per channel
// p < P and state n < NS:
//   dt_t,p = softplus(z_t,p + b_dt,p),  B_t = z_t[P .. P+NS),  C_t = z_t[P+NS .. P+2NS)
//   Abar_t,pn = exp(dt_t,p A_pn),  h_t,pn = Abar_t,pn h_t-1,pn + dt_t,p B_t,n xhat_t,p
//   y_t,p = xhat_t,p + sum_n C_t,n h_t,pn
// The gradient is the sum over token pairs of the VJPs of dl_t/dy_t lambda_{t,i},
// lambda_{t,i} = C_t prod_{j=i+1..t} A_j ([AS] Core claim, Proposition 2), summed per token
// i first: mu_i,pn = sum_t gy_t,p C_t,n prod_{j=i+1..t} Abar_j,pn over the window t - i < W,
// i.e. mu_i = e_i + Abar_{i+1} mu_{i+1} with e_i = gy_i,p C_i,n (full window), and blockwise
// mu^W_i = S_i + Q_i R(min(i+W-1, T-1)) for a window W (the same decomposition as the
// diagonal layer's: S, Q the reverse scan restarted at every block end, R the forward scan
// restarted at every block start, R(m) = sum_{t=s}^{m} e_t prod_{j=s+1..t} Abar_j).
//
// Work decomposition.  A thread owns one channel p and 8 of its states (SEL_NT); a CTA of
// 256 threads owns 256 / (NS / 8) channels of one chunk of TT consecutive tokens of one
// sequence and walks the chunk token by token.  Every scan runs in three launches with no
// CTA ever waiting on another: (1) each chunk's aggregate (the composite of its tokens),
// (2) one pass per (sequence, channel, state) over the chunk aggregates in scan order,
// writing each chunk's incoming carry in place, (3) each chunk again from its carry,
// writing the outputs.  The per-token inputs of the scans (z, xhat, gy: P + 2NS values a
// token) are small next to the state (P NS values), so reading them twice costs little;
// h is written once (forward) and read once (reverse).
#include <math.h>

#include "adj_internal.cuh"
#include "adj_sel.cuh"

namespace adj {

namespace {

constexpr int SEL_THREADS = 256;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float softplus_f(float z) { return z > 20.f ? z : log1pf(expf(z)); }
__device__ __forceinline__ float sigmoid_f(float z) { return 1.f / (1.f + expf(-z)); }
__device__ __forceinline__ float ldx(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ldx(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <int NS>
struct Geo {   // a thread's place: channel p, states n0 .. n0 + 8
    static constexpr int LP = NS / SEL_NT;               // threads per channel
    static constexpr int PC = SEL_THREADS / LP;          // channels per CTA
    int p, n0;
    bool act;
    __device__ Geo(int slice, int P) {
        p = slice * PC + int(threadIdx.x) / LP;
        n0 = (int(threadIdx.x) % LP) * SEL_NT;
        act = p < P;
    }
};

// 8 consecutive floats of a row (32-byte aligned)
__device__ __forceinline__ void ld8(const float *p, float (&v)[SEL_NT]) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(p)), b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st8(float *p, const float (&v)[SEL_NT]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void st8_stream(float *p, const float (&v)[SEL_NT]) {
    __stcs(reinterpret_cast<float4 *>(p), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
}

// Stage columns [col0, col0 + NS) of the chunk's z rows (B_t or C_t), zero past T.
template <int NS>
__device__ __forceinline__ void stage_cols(float (*dst)[NS], const float *z, int64_t row0, int64_t rows, int ZW,
                                           int col0, int TT) {
    for (int i = threadIdx.x; i < TT * NS; i += SEL_THREADS) {
        const int r = i / NS, n = i % NS;
        dst[r][n] = r < rows ? z[(row0 + r) * ZW + col0 + n] : 0.f;
    }
}

// ------------------------------------------------------------------ forward state scan
// MODE 0: aggregates (prod Abar, h at the chunk end from h = 0) -> aggX, aggY.
// MODE 1: outputs from the carries in aggY: h [B,T,P,NS] and y [B,T,P].
template <int NS, typename TX, int MODE>
__global__ void __launch_bounds__(SEL_THREADS) k_sel_fwd(const float *__restrict__ z, const TX *__restrict__ x,
                                                        const float *__restrict__ b_dt, const float *__restrict__ A,
                                                        float *__restrict__ aggX, float *__restrict__ aggY,
                                                        float *__restrict__ h, float *__restrict__ y, int64_t T, int P,
                                                        int TT, int64_t nchunks) {
    extern __shared__ float sm_sel[];
    float(*sB)[NS] = reinterpret_cast<float(*)[NS]>(sm_sel);
    float(*sC)[NS] = reinterpret_cast<float(*)[NS]>(sm_sel + TT * NS);
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const Geo<NS> g(int(blockIdx.y), P);
    const int ZW = P + 2 * NS;
    const int64_t c0 = c * TT, rows = (c0 + TT <= T ? TT : T - c0), row0 = b * T + c0;
    stage_cols<NS>(sB, z, row0, rows, ZW, P, TT);
    if (MODE == 1) stage_cols<NS>(sC, z, row0, rows, ZW, P + NS, TT);
    __syncthreads();
    // a channel's threads are adjacent lanes, so a warp's lanes past P are whole channels;
    // they stay in the loop (on channel 0's inputs, storing nothing) for the lane-pair sum
    const int pp = g.act ? g.p : 0;
    float A2[SEL_NT], st[SEL_NT], pr[SEL_NT];
#pragma unroll
    for (int k = 0; k < SEL_NT; ++k) {
        A2[k] = A[pp * NS + g.n0 + k] * LOG2E;
        pr[k] = 1.f;
    }
    const int64_t ai = ((b * nchunks + c) * P + pp) * NS + g.n0;
    if (MODE == 1) {
#pragma unroll
        for (int k = 0; k < SEL_NT; ++k) st[k] = aggY[ai + k];
    } else {
#pragma unroll
        for (int k = 0; k < SEL_NT; ++k) st[k] = 0.f;
    }
    const float bd = b_dt[pp];
    for (int r = 0; r < rows; ++r) {
        const int64_t row = row0 + r;
        const float dt = softplus_f(z[row * ZW + pp] + bd);
        const float xv = ldx(x + row * P + pp);
        const float dx = dt * xv;
        float yp = 0.f;
#pragma unroll
        for (int k = 0; k < SEL_NT; ++k) {
            const float ab = exp2f(dt * A2[k]);
            st[k] = fmaf(ab, st[k], dx * sB[r][g.n0 + k]);
            if (MODE == 0) pr[k] *= ab;
            else yp = fmaf(sC[r][g.n0 + k], st[k], yp);
        }
        if (MODE == 1) {
            if (g.act) st8_stream(h + (row * P + pp) * NS + g.n0, st);
            if (Geo<NS>::LP == 2) yp += __shfl_xor_sync(0xffffffffu, yp, 1);
            if (g.act && g.n0 == 0) y[row * P + pp] = xv + yp;
        }
    }
    if (MODE == 0 && g.act) {
        st8(aggX + ai, pr);
        st8(aggY + ai, st);
    }
}

// ------------------------------------------------------------------ window scan R (truncated mode)
// R(m) = sum_{t=s}^{m} e_t prod_{j=s+1..t} Abar_j within each block of W tokens (s its
// start), e = gy C.  MODE 0: aggregates (Pi, R of the chunk from (1, 0), the block start's
// Abar left out) -> aggX, aggY; MODE 1: R [B,T,P,NS] from the carries (Pi_in, R_in).
template <int NS, int MODE>
__global__ void __launch_bounds__(SEL_THREADS) k_sel_win(const float *__restrict__ z, const float *__restrict__ gy,
                                                        const float *__restrict__ b_dt, const float *__restrict__ A,
                                                        float *__restrict__ aggX, float *__restrict__ aggY,
                                                        float *__restrict__ R, int64_t T, int P, int TT,
                                                        int64_t nchunks, int64_t W) {
    extern __shared__ float sm_sel[];
    float(*sC)[NS] = reinterpret_cast<float(*)[NS]>(sm_sel);
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const Geo<NS> g(int(blockIdx.y), P);
    const int ZW = P + 2 * NS;
    const int64_t c0 = c * TT, rows = (c0 + TT <= T ? TT : T - c0), row0 = b * T + c0;
    stage_cols<NS>(sC, z, row0, rows, ZW, P + NS, TT);
    __syncthreads();
    if (!g.act) return;
    float A2[SEL_NT], pi[SEL_NT], rr[SEL_NT];
    const int64_t ai = ((b * nchunks + c) * P + g.p) * NS + g.n0;
#pragma unroll
    for (int k = 0; k < SEL_NT; ++k) {
        A2[k] = A[g.p * NS + g.n0 + k] * LOG2E;
        pi[k] = MODE == 1 ? aggX[ai + k] : 1.f;
        rr[k] = MODE == 1 ? aggY[ai + k] : 0.f;
    }
    const float bd = b_dt[g.p];
    for (int r = 0; r < rows; ++r) {
        const int64_t row = row0 + r;
        const float gv = gy[row * P + g.p];
        if ((c0 + r) % W != 0) {
            const float dt = softplus_f(z[row * ZW + g.p] + bd);
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) pi[k] *= exp2f(dt * A2[k]);
        }
#pragma unroll
        for (int k = 0; k < SEL_NT; ++k) rr[k] = fmaf(pi[k], gv * sC[r][g.n0 + k], rr[k]);
        if (MODE == 1) st8(R + (row * P + g.p) * NS + g.n0, rr);
    }
    if (MODE == 0) {
        st8(aggX + ai, pi);
        st8(aggY + ai, rr);
    }
}

// ------------------------------------------------------------------ carries over chunks
// One thread per (sequence, channel-state); walks the chunk aggregates in scan order and
// writes every chunk's incoming carry over its aggregate (X, Y in place).
//   KIND 0 forward h:   h_in(0) = 0;  h_in(c+1) = X_c h_in(c) + Y_c             -> Y = h_in
//   KIND 1 reverse mu:  from the last chunk down; (q, m) = (1, 0) where the chunk ends a
//                       block or the sequence; (q, m)(c-1) = (X_c q, X_c m + Y_c) -> X = q, Y = m
//   KIND 2 window R:    (pi, r) = (1, 0) where the chunk starts a block;
//                       (pi, r)(c+1) = (pi X_c, r + pi Y_c)                    -> X = pi, Y = r
// The loads run PF chunks ahead of the dependent chain.
template <int KIND>
__global__ void __launch_bounds__(256) k_sel_carry(float *__restrict__ X, float *__restrict__ Y, int64_t B,
                                                  int64_t PN, int64_t nchunks, int64_t T, int TT, int64_t W) {
    constexpr int PF = 8;
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= B * PN) return;
    const int64_t b = i / PN, j = i % PN;
    const int64_t base = b * nchunks * PN + j;
    float q = 1.f, m = 0.f;
    for (int64_t s = 0; s < nchunks; s += PF) {
        float xv[PF], yv[PF];
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            const int64_t c = KIND == 1 ? nchunks - 1 - (s + u) : s + u;
            if (s + u < nchunks) {
                xv[u] = X[base + c * PN];
                yv[u] = Y[base + c * PN];
            }
        }
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            if (s + u >= nchunks) break;
            const int64_t c = KIND == 1 ? nchunks - 1 - (s + u) : s + u;
            const int64_t at = base + c * PN;
            if (KIND == 0) {
                Y[at] = m;
                m = fmaf(xv[u], m, yv[u]);
            } else if (KIND == 1) {
                const int64_t c1 = (c + 1) * TT < T ? (c + 1) * TT : T;
                if (c1 % W == 0 || c1 >= T) {
                    q = 1.f;
                    m = 0.f;
                }
                X[at] = q;
                Y[at] = m;
                m = fmaf(xv[u], m, yv[u]);
                q *= xv[u];
            } else {
                if ((c * TT) % W == 0) {
                    q = 1.f;
                    m = 0.f;
                }
                X[at] = q;
                Y[at] = m;
                m = fmaf(q, yv[u], m);
                q *= xv[u];
            }
        }
    }
}

// ------------------------------------------------------------------ reverse adjoint scan + VJPs
// Butterfly transpose-sum over the lanes whose bit `lb` and above index the channel: each
// of the 2 SEL_NT values v[] ends summed over the 32 / LP channels of the warp, one value
// per lane (lane l holds value idx(l)).
template <int LP>
__device__ __forceinline__ float warp_tsum16(float (&v)[2 * SEL_NT], int lane) {
    // levels over lane bits 4..1, the 16 values halving each level; with LP == 1 the lane
    // pairs (bit 0) are summed last
    constexpr int V = 2 * SEL_NT;
    int cnt = V;
#pragma unroll
    for (int bit = 4; bit >= 1; --bit) {
        const int s = 1 << bit;
        const bool up = (lane & s) != 0;
        cnt >>= 1;
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
            if (i < cnt) {
                const float send = up ? v[i] : v[i + cnt];
                const float keep = up ? v[i + cnt] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
            }
        }
    }
    float r = v[0];
    if (LP == 1) r += __shfl_xor_sync(0xffffffffu, r, 1);
    return r;
}
// the value index lane l holds after warp_tsum16
__device__ __forceinline__ int tsum_index(int lane) {
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// MODE 0: chunk aggregates of the reverse scan (Q = prod_{c0 < j <= c1} Abar_j, S = mu_c0
// from mu_c1 = 0) -> aggX, aggY.
// MODE 1: outputs from the carries (q_in, mu_in) in aggX, aggY: dz[:, :P] (the dt part,
// through the softplus), the CTA's partial sums over its channels of dB and dC per token
// -> bc [B*T, nslices, 2 NS], and the chunk's dA partial -> dAp [B*nchunks, P, NS].
// TRUNC: mu^W = mu + q R(min(t+W-1, T-1)) where a later block exists and t starts none.
template <int NS, typename TX, typename TD, int MODE, bool TRUNC>
__global__ void __launch_bounds__(SEL_THREADS) k_sel_bwd(const float *__restrict__ z, const TX *__restrict__ x,
                                                        const float *__restrict__ gy, const float *__restrict__ h,
                                                        const float *__restrict__ R, const float *__restrict__ b_dt,
                                                        const float *__restrict__ A, float *__restrict__ aggX,
                                                        float *__restrict__ aggY, TD *__restrict__ dz,
                                                        float *__restrict__ bc, float *__restrict__ dAp, int64_t T,
                                                        int P, int TT, int64_t nchunks, int nslices, int64_t W) {
    extern __shared__ float sm_sel[];
    constexpr int LP = Geo<NS>::LP;
    constexpr int TB = 16;   // tokens per batch of the cross-warp sums
    float(*sB)[NS] = reinterpret_cast<float(*)[NS]>(sm_sel);
    float(*sC)[NS] = reinterpret_cast<float(*)[NS]>(sm_sel + TT * NS);
    float(*sW)[TB][32] = reinterpret_cast<float(*)[TB][32]>(sm_sel + 2 * TT * NS);   // [8 warps]
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int slice = int(blockIdx.y);
    const Geo<NS> g(slice, P);
    const int ZW = P + 2 * NS, lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    const int64_t c0 = c * TT, rows = (c0 + TT <= T ? TT : T - c0), row0 = b * T + c0;
    if (MODE == 1) stage_cols<NS>(sB, z, row0, rows, ZW, P, TT);
    stage_cols<NS>(sC, z, row0, rows, ZW, P + NS, TT);
    __syncthreads();
    const int pp = g.act ? g.p : 0;   // inactive threads run the loop (the warp sums need them) on zeros
    float A2[SEL_NT], mu[SEL_NT], q[SEL_NT], abn[SEL_NT], dA[SEL_NT], hc[SEL_NT];
    const int64_t ai = ((b * nchunks + c) * P + pp) * NS + g.n0;
    const float bd = b_dt[pp];
    // Abar of the token after the chunk (0 past the sequence end)
    float dtn = 0.f;
    const bool has_next = c0 + rows < T;
    if (has_next) dtn = softplus_f(z[(row0 + rows) * ZW + pp] + bd);
#pragma unroll
    for (int k = 0; k < SEL_NT; ++k) {
        A2[k] = A[pp * NS + g.n0 + k] * LOG2E;
        abn[k] = has_next ? exp2f(dtn * A2[k]) : 0.f;
        mu[k] = MODE == 1 && g.act ? aggY[ai + k] : 0.f;
        q[k] = MODE == 1 && g.act ? aggX[ai + k] : 1.f;
        dA[k] = 0.f;
    }
    if (MODE == 1) {
        if (g.act) ld8(h + ((row0 + rows - 1) * P + pp) * NS + g.n0, hc);
        else
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) hc[k] = 0.f;
    }
    const bool next_block = TRUNC && (c0 / W + 1) * W < T;
    for (int r = int(rows) - 1; r >= 0; --r) {
        const int64_t t = c0 + r, row = row0 + r;
        const float gv = g.act ? gy[row * P + pp] : 0.f;
        const float zr = z[row * ZW + pp] + bd;
        const float dt = softplus_f(zr);
        float ab[SEL_NT];
#pragma unroll
        for (int k = 0; k < SEL_NT; ++k) {
            mu[k] = fmaf(abn[k], mu[k], gv * sC[r][g.n0 + k]);
            if (MODE == 0 || TRUNC) q[k] *= abn[k];   // MODE 0: the aggregate's product
            ab[k] = exp2f(dt * A2[k]);
        }
        if (MODE == 1) {
            float mw[SEL_NT];
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) mw[k] = mu[k];
            if (TRUNC && next_block && t % W != 0 && g.act) {
                const int64_t m = t + W - 1 < T - 1 ? t + W - 1 : T - 1;
                float rv[SEL_NT];
                ld8(R + ((b * T + m) * P + pp) * NS + g.n0, rv);
#pragma unroll
                for (int k = 0; k < SEL_NT; ++k) mw[k] = fmaf(q[k], rv[k], mw[k]);
            }
            // h_{t-1}
            float hp[SEL_NT];
            if (t > 0 && g.act) ld8(h + ((row - 1) * P + pp) * NS + g.n0, hp);
            else
#pragma unroll
                for (int k = 0; k < SEL_NT; ++k) hp[k] = 0.f;
            const float xv = g.act ? ldx(x + row * P + pp) : 0.f;
            float ddt = 0.f, v[2 * SEL_NT];
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) {
                const float aah = ab[k] * hp[k];
                ddt = fmaf(mw[k], fmaf(A2[k], aah * (1.f / LOG2E), sB[r][g.n0 + k] * xv), ddt);
                dA[k] = fmaf(mw[k] * dt, aah, dA[k]);
                v[k] = mw[k] * dt * xv;          // dB_t,n share
                v[SEL_NT + k] = gv * hc[k];      // dC_t,n share
                hc[k] = hp[k];
            }
            if (LP == 2) ddt += __shfl_xor_sync(0xffffffffu, ddt, 1);
            if (g.act && g.n0 == 0) {
                const float val = ddt * sigmoid_f(zr);
                if constexpr (sizeof(TD) == 2) dz[row * ZW + pp] = __float2bfloat16_rn(val);
                else dz[row * ZW + pp] = val;
            }
            // per-token sums over the CTA's channels: warp butterfly, then the 8 warps in
            // order, TB tokens a batch
            const float wsum = warp_tsum16<LP>(v, lane);
            const int slot = r % TB;
            sW[wp][slot][lane] = wsum;
            if (slot == 0 || r == 0) {
                __syncthreads();
                const int nb = TB - slot;   // tokens of this batch: rows r .. r + nb - 1 ... clipped
                for (int e = threadIdx.x; e < TB * 32; e += SEL_THREADS) {
                    const int s2 = e / 32, l = e % 32;
                    if (s2 < slot || s2 >= slot + nb || r + (s2 - slot) >= rows) continue;
                    float acc = 0.f;
#pragma unroll
                    for (int w8 = 0; w8 < SEL_THREADS / 32; ++w8) acc += sW[w8][s2][l];
                    // lane l's value index: n-block (LP == 2: lane bit 0) and tsum index
                    const int vi = tsum_index(l);
                    const int nblk = LP == 2 ? (l & 1) : 0;
                    const int which = vi >> 3, n = nblk * SEL_NT + (vi & 7);
                    if (LP == 1 && (l & 1)) continue;   // duplicate of lane l - 1
                    const int64_t trow = row0 + r + (s2 - slot);
                    bc[(trow * nslices + slice) * (2 * NS) + which * NS + n] = acc;
                }
                __syncthreads();
            }
        }
#pragma unroll
        for (int k = 0; k < SEL_NT; ++k) abn[k] = ab[k];
    }
    if (!g.act) return;
    if (MODE == 0) {
        st8(aggX + ai, q);
        st8(aggY + ai, mu);
    } else {
        st8(dAp + ((b * nchunks + c) * P + g.p) * NS + g.n0, dA);
    }
}

// dz[:, P + j] = sum over slices of bc (j < 2 NS), in the dz storage type.
template <typename TD>
__global__ void k_sel_bc_reduce(const float *__restrict__ bc, TD *__restrict__ dz, int64_t rows, int P, int NS2,
                                int nslices) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * NS2) return;
    const int64_t r = i / NS2;
    const int j = int(i % NS2);
    float acc = 0.f;
    for (int s = 0; s < nslices; ++s) acc += bc[(r * nslices + s) * NS2 + j];
    if constexpr (sizeof(TD) == 2) dz[r * (P + NS2) + P + j] = __float2bfloat16_rn(acc);
    else dz[r * (P + NS2) + P + j] = acc;
}

// dA[j] = sum over parts (rows of dAp) in order.
__global__ void k_sel_rows_sum(const float *__restrict__ part, float *__restrict__ out, int64_t nparts, int64_t n) {
    const int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= n) return;
    float acc = 0.f;
    for (int64_t s = 0; s < nparts; ++s) acc += part[s * n + j];
    out[j] = acc;
}

// db_dt partials: part[blk][p] = sum over block blk's rows of dz[:, p] (row stride ld)
template <typename TD>
__global__ void k_sel_colsum(const TD *__restrict__ dz, int64_t rows, int P, int ld, int nblk,
                             float *__restrict__ part) {
    const int p = int(blockIdx.x) * blockDim.x + threadIdx.x;
    const int blk = int(blockIdx.y);
    if (p >= P) return;
    const int64_t r0 = rows * blk / nblk, r1 = rows * (blk + 1) / nblk;
    float acc = 0.f;
    for (int64_t r = r0; r < r1; ++r) {
        if constexpr (sizeof(TD) == 2) acc += __bfloat162float(dz[r * ld + p]);
        else acc += dz[r * ld + p];
    }
    part[int64_t(blk) * P + p] = acc;
}

template <class K>
cudaError_t smem_attr(K kern, size_t smem) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

}  // namespace

// ============================================================================ launchers
int sel_chunk(int64_t T, int64_t W) {
    int tt = SEL_TT_MAX;
    if (W > 0 && W < T)
        while (tt > SEL_TT_MIN && W % tt) tt >>= 1;
    return tt;
}
bool sel_window_ok(int64_t T, int64_t W) { return W <= 0 || W >= T || W % SEL_TT_MIN == 0; }
int sel_slices(int P, int NS) { return int((P + SEL_THREADS / (NS / SEL_NT) - 1) / (SEL_THREADS / (NS / SEL_NT))); }

static dim3 sel_grid(int64_t B, int64_t nchunks, int P, int NS) {
    return dim3(unsigned(nchunks), unsigned(sel_slices(P, NS)), unsigned(B));
}

template <int NS, typename TX>
static cudaError_t sel_fwd_t(const float *z, const void *x, const float *b_dt, const float *A, float *h, float *y,
                             float *aggX, float *aggY, int64_t B, int64_t T, int P, cudaStream_t st) {
    const int TT = sel_chunk(T, 0);
    const int64_t nchunks = (T + TT - 1) / TT;
    const dim3 grid = sel_grid(B, nchunks, P, NS);
    const size_t smem = size_t(2) * TT * NS * 4;
    const TX *xt = static_cast<const TX *>(x);
    cudaError_t e;
    if ((e = smem_attr(k_sel_fwd<NS, TX, 0>, smem)) != cudaSuccess) return e;
    if ((e = smem_attr(k_sel_fwd<NS, TX, 1>, smem)) != cudaSuccess) return e;
    k_sel_fwd<NS, TX, 0><<<grid, SEL_THREADS, smem, st>>>(z, xt, b_dt, A, aggX, aggY, h, y, T, P, TT, nchunks);
    const int64_t n = B * int64_t(P) * NS;
    k_sel_carry<0><<<unsigned((n + 255) / 256), 256, 0, st>>>(aggX, aggY, B, int64_t(P) * NS, nchunks, T, TT, T);
    k_sel_fwd<NS, TX, 1><<<grid, SEL_THREADS, smem, st>>>(z, xt, b_dt, A, aggX, aggY, h, y, T, P, TT, nchunks);
    return cudaGetLastError();
}

cudaError_t launch_sel_fwd(const float *z, const void *x, bool x_bf16, const float *b_dt, const float *A, float *h,
                           float *y, float *aggX, float *aggY, int64_t B, int64_t T, int P, int NS, cudaStream_t st) {
    if (NS == 16) return x_bf16 ? sel_fwd_t<16, __nv_bfloat16>(z, x, b_dt, A, h, y, aggX, aggY, B, T, P, st)
                                : sel_fwd_t<16, float>(z, x, b_dt, A, h, y, aggX, aggY, B, T, P, st);
    if (NS == 8) return x_bf16 ? sel_fwd_t<8, __nv_bfloat16>(z, x, b_dt, A, h, y, aggX, aggY, B, T, P, st)
                               : sel_fwd_t<8, float>(z, x, b_dt, A, h, y, aggX, aggY, B, T, P, st);
    return cudaErrorInvalidValue;
}

template <int NS, typename TX, typename TD>
static cudaError_t sel_bwd_t(const float *z, const void *x, const float *gy, const float *h, const float *b_dt,
                             const float *A, void *dz, float *dA, const SelBwdWs &w, int64_t B, int64_t T, int P,
                             int64_t W, cudaStream_t st) {
    const bool trunc = W > 0 && W < T;
    const int TT = sel_chunk(T, trunc ? W : 0);
    const int64_t nchunks = (T + TT - 1) / TT, Wk = trunc ? W : T;
    const int nsl = sel_slices(P, NS);
    const dim3 grid = sel_grid(B, nchunks, P, NS);
    const int64_t n = B * int64_t(P) * NS;
    const unsigned cgrid = unsigned((n + 255) / 256);
    const TX *xt = static_cast<const TX *>(x);
    TD *dzt = static_cast<TD *>(dz);
    cudaError_t e;
    if (trunc) {
        const size_t sm1 = size_t(TT) * NS * 4;
        if ((e = smem_attr(k_sel_win<NS, 0>, sm1)) != cudaSuccess) return e;
        if ((e = smem_attr(k_sel_win<NS, 1>, sm1)) != cudaSuccess) return e;
        k_sel_win<NS, 0><<<grid, SEL_THREADS, sm1, st>>>(z, gy, b_dt, A, w.winX, w.winY, w.R, T, P, TT, nchunks, Wk);
        k_sel_carry<2><<<cgrid, 256, 0, st>>>(w.winX, w.winY, B, int64_t(P) * NS, nchunks, T, TT, Wk);
        k_sel_win<NS, 1><<<grid, SEL_THREADS, sm1, st>>>(z, gy, b_dt, A, w.winX, w.winY, w.R, T, P, TT, nchunks, Wk);
    }
    const size_t sm = size_t(2) * TT * NS * 4 + size_t(SEL_THREADS / 32) * 16 * 32 * 4;
#define ADJ_SEL_BWD(TR)                                                                                            \
    do {                                                                                                           \
        if ((e = smem_attr(k_sel_bwd<NS, TX, TD, 0, TR>, sm)) != cudaSuccess) return e;                            \
        if ((e = smem_attr(k_sel_bwd<NS, TX, TD, 1, TR>, sm)) != cudaSuccess) return e;                            \
        k_sel_bwd<NS, TX, TD, 0, TR><<<grid, SEL_THREADS, sm, st>>>(z, xt, gy, h, w.R, b_dt, A, w.aggX, w.aggY,    \
                                                                    dzt, w.bc, w.dAp, T, P, TT, nchunks, nsl, Wk); \
        k_sel_carry<1><<<cgrid, 256, 0, st>>>(w.aggX, w.aggY, B, int64_t(P) * NS, nchunks, T, TT, Wk);             \
        k_sel_bwd<NS, TX, TD, 1, TR><<<grid, SEL_THREADS, sm, st>>>(z, xt, gy, h, w.R, b_dt, A, w.aggX, w.aggY,    \
                                                                    dzt, w.bc, w.dAp, T, P, TT, nchunks, nsl, Wk); \
    } while (0)
    if (trunc) ADJ_SEL_BWD(true);
    else ADJ_SEL_BWD(false);
#undef ADJ_SEL_BWD
    const int64_t nbc = B * T * 2 * NS;
    k_sel_bc_reduce<TD><<<unsigned((nbc + 255) / 256), 256, 0, st>>>(w.bc, dzt, B * T, P, 2 * NS, nsl);
    k_sel_rows_sum<<<unsigned((int64_t(P) * NS + 255) / 256), 256, 0, st>>>(w.dAp, dA, B * nchunks,
                                                                          int64_t(P) * NS);
    return cudaGetLastError();
}

cudaError_t launch_sel_bwd(const float *z, const void *x, bool x_bf16, const float *gy, const float *h,
                           const float *b_dt, const float *A, void *dz, bool d_bf16, float *dA, const SelBwdWs &w,
                           int64_t B, int64_t T, int P, int NS, int64_t W, cudaStream_t st) {
#define ADJ_SEL_B(NSV)                                                                                              \
    do {                                                                                                            \
        if (x_bf16) {                                                                                               \
            if (d_bf16) return sel_bwd_t<NSV, __nv_bfloat16, __nv_bfloat16>(z, x, gy, h, b_dt, A, dz, dA, w, B, T, P, W, st); \
            return sel_bwd_t<NSV, __nv_bfloat16, float>(z, x, gy, h, b_dt, A, dz, dA, w, B, T, P, W, st);          \
        }                                                                                                           \
        if (d_bf16) return sel_bwd_t<NSV, float, __nv_bfloat16>(z, x, gy, h, b_dt, A, dz, dA, w, B, T, P, W, st);   \
        return sel_bwd_t<NSV, float, float>(z, x, gy, h, b_dt, A, dz, dA, w, B, T, P, W, st);                       \
    } while (0)
    if (NS == 16) ADJ_SEL_B(16);
    if (NS == 8) ADJ_SEL_B(8);
#undef ADJ_SEL_B
    return cudaErrorInvalidValue;
}

cudaError_t launch_sel_colsum(const void *dz, bool d_bf16, int64_t rows, int P, int ld, int nblk, float *part,
                              cudaStream_t st) {
    const dim3 grid(unsigned((P + 127) / 128), unsigned(nblk));
    if (d_bf16)
        k_sel_colsum<__nv_bfloat16><<<grid, 128, 0, st>>>(static_cast<const __nv_bfloat16 *>(dz), rows, P, ld, nblk, part);
    else
        k_sel_colsum<float><<<grid, 128, 0, st>>>(static_cast<const float *>(dz), rows, P, ld, nblk, part);
    return cudaGetLastError();
}

}  // namespace adj
