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
// Work decomposition.  A thread owns one channel p and SEL_NT = 8 of its states; a CTA of
// 256 threads owns 256 / (NS / 8) channels of one chunk of TT consecutive tokens of one
// sequence and walks the chunk token by token.  Every scan runs in three launches with no
// CTA ever waiting on another: (1) each chunk's aggregate (the composite of its tokens),
// (2) one pass per (sequence, channel, state) over the chunk aggregates in scan order,
// writing each chunk's incoming carry in place, (3) each chunk again from its carry,
// writing the outputs.  The per-token inputs (the step dt = softplus(z + b_dt), xhat, gy,
// B_t, C_t: P + 2NS values a token) are staged in shared memory a sub-chunk at a time by
// coalesced loads of the whole CTA, so the per-token walk reads only shared memory; they
// are small next to the state (P NS values a token), so reading them in both passes costs
// little.  h is written once (forward, streaming stores) and read once (reverse): the
// reverse pass has one more warp that only brings the chunk's state rows (and, truncated,
// the window sums R) into a ring of shared-memory stages by bulk copies, counted on a
// "full" mbarrier per stage; the walking warps release a stage on its "empty" mbarrier
// (bounded waits on both).
#include <math.h>

#include "adj_internal.cuh"
#include "adj_ptx.cuh"
#include "adj_sel.cuh"

namespace adj {

namespace {

constexpr int SEL_THREADS = 256;   // the walking threads of a CTA
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float softplus_f(float z) { return z > 20.f ? z : log1pf(expf(z)); }
__device__ __forceinline__ float ldx(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ldx(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
// 2^x by the SFU's approximate exponential (relative error about 2^-22; subnormal results
// flush to zero, a decay that small is zero for every purpose here)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// barrier 1 among the CTA's 256 walking threads
__device__ __forceinline__ void walkers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int NS>
struct Geo {   // a thread's place: channel p (q within the slice), states n0 .. n0 + SEL_NT
    static constexpr int LP = NS / SEL_NT;               // threads a channel (adjacent lanes)
    static constexpr int PC = SEL_THREADS / LP;          // channels a CTA
    static constexpr int SC = 2048 / PC;                 // tokens a staged sub-chunk
    int q, p, n0;
    bool act;
    __device__ Geo(int slice, int P) {
        q = int(threadIdx.x) / LP;
        p = slice * PC + q;
        n0 = (int(threadIdx.x) % LP) * SEL_NT;
        act = p < P;
    }
};

// two floats as bf16 (round to nearest even), the first in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// sum over the LP lanes of a channel
template <int LP>
__device__ __forceinline__ float chan_sum(float v) {
    if (LP >= 2) v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

__device__ __forceinline__ void ld8s(const float *p, float (&v)[SEL_NT]) {   // shared
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ld8g(const float *p, float (&v)[SEL_NT]) {   // global, L2
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p)), b = __ldcg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st8v(float *p, const float (&v)[SEL_NT]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void st8s(float *p, const float (&v)[SEL_NT]) {   // streaming
    __stcs(reinterpret_cast<float4 *>(p), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
}

// Shared staging of one sub-chunk (rows [r0, r0 + nr) of the chunk starting at global row
// row0; zero past nr and past P): dt [SC][PC], xhat [SC][PC] (WX), gy [SC][PC] (WG), and
// the z columns of B_t and C_t [SC][NS] each.
template <int NS>
struct Stage {
    float *dt, *x, *g, *sig, *B, *C, *zr;
};
// wz: also the raw z of the dt columns (the reverse pass's input path)
template <int NS>
__device__ __forceinline__ Stage<NS> stage_carve(float *base, bool wz = false) {
    constexpr int PC = Geo<NS>::PC, SC = Geo<NS>::SC;
    Stage<NS> s;
    s.dt = base;
    s.x = s.dt + SC * PC;
    s.g = s.x + SC * PC;
    s.sig = s.g + SC * PC;
    s.B = s.sig + SC * PC;
    s.C = s.B + SC * NS;
    s.zr = wz ? s.C + SC * NS : nullptr;
    return s;
}
template <int NS>
constexpr size_t stage_floats(bool wz = false) {
    return size_t(Geo<NS>::SC) * Geo<NS>::PC * (wz ? 5 : 4) + size_t(Geo<NS>::SC) * NS * 2;
}
// The sub-chunk's per-token inputs as loaded into registers (a thread's share).
template <int NS>
struct StageRegs {
    static constexpr int PER = Geo<NS>::SC * Geo<NS>::PC / SEL_THREADS;
    float z[PER], x[PER], g[PER], b[PER], bc[(Geo<NS>::SC * 2 * NS + SEL_THREADS - 1) / SEL_THREADS];
};
template <int NS, typename TX, bool WX, bool WG>
__device__ __forceinline__ void stage_load(StageRegs<NS> &R, const float *__restrict__ z, const TX *__restrict__ x,
                                           const float *__restrict__ gy, const float *__restrict__ b_dt, int P,
                                           int ZW, int64_t row0, int r0, int nr, int p0) {
    constexpr int PC = Geo<NS>::PC, SC = Geo<NS>::SC, PER = StageRegs<NS>::PER;
#pragma unroll
    for (int u = 0; u < PER; ++u) {   // every load of the sub-chunk in flight at once
        const int i = int(threadIdx.x) + u * SEL_THREADS, r = i / PC, p = p0 + i % PC;
        const bool ok = r < nr && p < P;
        const int64_t row = row0 + r0 + r;
        R.z[u] = ok ? z[row * ZW + p] : 0.f;
        R.b[u] = ok ? __ldg(b_dt + p) : 0.f;
        R.x[u] = (WX && ok) ? ldx(x + row * P + p) : 0.f;
        R.g[u] = (WG && ok) ? gy[row * P + p] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < int(sizeof(R.bc) / sizeof(float)); ++u) {
        const int i = int(threadIdx.x) + u * SEL_THREADS, r = i / (2 * NS), j = i % (2 * NS);
        R.bc[u] = (i < SC * 2 * NS && r < nr) ? z[(row0 + r0 + r) * ZW + P + j] : 0.f;
    }
}
template <int NS, bool WX, bool WG, bool WZ = false>
__device__ __forceinline__ void stage_store(const Stage<NS> &s, const StageRegs<NS> &R, int nr, int p0, int P) {
    constexpr int PC = Geo<NS>::PC, SC = Geo<NS>::SC, PER = StageRegs<NS>::PER;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int i = int(threadIdx.x) + u * SEL_THREADS, r = i / PC, p = p0 + i % PC;
        const bool ok = r < nr && p < P;
        // dt = softplus(s) and, for the reverse pass, sigmoid(s) = e^s / (1 + e^s), s = z + b_dt
        const float sv = R.z[u] + R.b[u], es = expf(fminf(sv, 20.f));
        s.dt[i] = ok ? (sv > 20.f ? sv : log1pf(es)) : 0.f;
        if (WG) s.sig[i] = ok ? es / (1.f + es) : 0.f;
        if (WX) s.x[i] = R.x[u];
        if (WG) s.g[i] = R.g[u];
        if (WZ) s.zr[i] = ok ? R.z[u] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < int(sizeof(R.bc) / sizeof(float)); ++u) {
        const int i = int(threadIdx.x) + u * SEL_THREADS, r = i / (2 * NS), j = i % (2 * NS);
        if (i < SC * 2 * NS) {
            if (j < NS) s.B[r * NS + j] = R.bc[u];
            else s.C[r * NS + j - NS] = R.bc[u];
        }
    }
}
// L2 prefetch of a sub-chunk's per-token inputs (rows [r0, r0 + nr) of the chunk at row0,
// this CTA's channels): z's dt columns, xhat and gy a 128-byte line a thread-step, and the
// row's B and C columns; only addresses inside the arrays.
template <int NS, typename TX>
__device__ __forceinline__ void stage_prefetch(const float *__restrict__ z, const TX *__restrict__ x,
                                               const float *__restrict__ gy, int P, int ZW, int64_t row0, int r0,
                                               int nr, int p0) {
    constexpr int PC = Geo<NS>::PC;
    constexpr int LZ = PC * 4 / 128, LX = PC * int(sizeof(TX)) / 128;   // lines a row
    constexpr int PER_ROW = 2 * LZ + LX + 1;                            // z, gy, xhat, B|C
    const int pw = P - p0 < PC ? P - p0 : PC;
    for (int e = int(threadIdx.x); e < nr * PER_ROW; e += SEL_THREADS) {
        const int r = e / PER_ROW, k = e % PER_ROW;
        const int64_t row = row0 + r0 + r;
        const void *a;
        if (k < LZ) {
            if (k * 32 >= pw) continue;
            a = z + row * ZW + p0 + k * 32;
        } else if (k < 2 * LZ) {
            if ((k - LZ) * 32 >= pw) continue;
            a = gy + row * P + p0 + (k - LZ) * 32;
        } else if (k < 2 * LZ + LX) {
            if ((k - 2 * LZ) * (128 / int(sizeof(TX))) >= pw) continue;
            a = x + row * P + p0 + (k - 2 * LZ) * (128 / int(sizeof(TX)));
        } else {
            a = z + row * ZW + P;
        }
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
}

template <int NS, typename TX, bool WX, bool WG, bool WZ = false>
__device__ __forceinline__ void stage_sub(const Stage<NS> &s, const float *__restrict__ z, const TX *__restrict__ x,
                                          const float *__restrict__ gy, const float *__restrict__ b_dt, int P,
                                          int ZW, int64_t row0, int r0, int nr, int p0) {
    StageRegs<NS> R;
    stage_load<NS, TX, WX, WG>(R, z, x, gy, b_dt, P, ZW, row0, r0, nr, p0);
    stage_store<NS, WX, WG, WZ>(s, R, nr, p0, P);
}

// ------------------------------------------------------------------ forward state scan
// Forward and window scans run three CTAs an SM (80 registers a thread; four, at 64, spill),
// except the forward output pass of a stacked layer (residual input), which ran slower so.
// MODE 0: aggregates (prod Abar, h at the chunk end from h = 0) -> aggX, aggY.
// MODE 1: outputs from the carries in aggY: h [B,T,P,NS] and y = xres + sum_n C h [B,T,P]
// (XR: the residual input xres, staged with the other per-token inputs; else xhat's values).
template <int NS, typename TX, int MODE, bool XR = false>
__global__ void __launch_bounds__(SEL_THREADS, XR ? 2 : 3) k_sel_fwd(const float *__restrict__ z, const TX *__restrict__ x,
                                                        const float *__restrict__ b_dt, const float *__restrict__ A,
                                                        float *__restrict__ aggX, float *__restrict__ aggY,
                                                        float *__restrict__ h, float *__restrict__ y,
                                                        const float *__restrict__ xres, int64_t T, int P, int TT,
                                                        int64_t nchunks) {
    extern __shared__ __align__(16) float sm_sel[];
    constexpr int PC = Geo<NS>::PC, LP = Geo<NS>::LP, SC = Geo<NS>::SC;
    const Stage<NS> sg = stage_carve<NS>(sm_sel);
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int slice = int(blockIdx.y);
    const Geo<NS> g(slice, P);
    const int ZW = P + 2 * NS;
    const int64_t c0 = c * TT, row0 = b * T + c0;
    const int rows = int(c0 + TT <= T ? TT : T - c0);
    // a channel's lanes past P stay in the walk (on zeros, storing nothing) for the lane sums
    const int pp = g.act ? g.p : 0;
    float A2[SEL_NT], st[SEL_NT], pr[SEL_NT];
#pragma unroll
    for (int k = 0; k < SEL_NT; ++k) {
        A2[k] = A[pp * NS + g.n0 + k] * LOG2E;
        pr[k] = 1.f;
        st[k] = 0.f;
    }
    const int64_t ai = ((b * nchunks + c) * P + pp) * NS + g.n0;
    if (MODE == 1 && g.act) ld8g(aggY + ai, st);
    // the next sub-chunk's inputs load into registers while this one is walked
    StageRegs<NS> R;   // (XR: xres rides in the slot of gy, which the forward pass does not use)
    stage_load<NS, TX, true, XR>(R, z, x, xres, b_dt, P, ZW, row0, 0, rows < SC ? rows : SC, slice * PC);
    for (int r0 = 0; r0 < rows; r0 += SC) {
        const int nr = rows - r0 < SC ? rows - r0 : SC;
        __syncthreads();   // the previous sub-chunk is consumed
        stage_store<NS, true, XR>(sg, R, nr, slice * PC, P);
        __syncthreads();
        if (r0 + SC < rows) {
            const int nn = rows - r0 - SC < SC ? rows - r0 - SC : SC;
            stage_load<NS, TX, true, XR>(R, z, x, xres, b_dt, P, ZW, row0, r0 + SC, nn, slice * PC);
        }
        for (int r = 0; r < nr; ++r) {
            const float dt = sg.dt[r * PC + g.q], xv = sg.x[r * PC + g.q], dx = dt * xv;
            float Bv[SEL_NT], Cv[SEL_NT];
            ld8s(sg.B + r * NS + g.n0, Bv);
            if (MODE == 1) ld8s(sg.C + r * NS + g.n0, Cv);
            float yp = 0.f;
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) {
                const float ab = ex2(dt * A2[k]);
                st[k] = fmaf(ab, st[k], dx * Bv[k]);
                if (MODE == 0) pr[k] *= ab;
                else yp = fmaf(Cv[k], st[k], yp);
            }
            if (MODE == 1) {
                const int64_t row = row0 + r0 + r;
                if (g.act) st8s(h + (row * P + pp) * NS + g.n0, st);
                yp = chan_sum<LP>(yp);
                if (g.act && g.n0 == 0) y[row * P + pp] = (XR ? sg.g[r * PC + g.q] : xv) + yp;
            }
        }
    }
    if (MODE == 0 && g.act) {
        st8v(aggX + ai, pr);
        st8v(aggY + ai, st);
    }
}

// ------------------------------------------------------------------ window scan R (truncated mode)
// R(m) = sum_{t=s}^{m} e_t prod_{j=s+1..t} Abar_j within each block of W tokens (s its
// start), e = gy C.  MODE 1: R [B,T,P,NS] from the carries (Pi_in, R_in) in aggX, aggY.
// MODE 0: both scans' chunk aggregates in one forward walk.  With Pc = prod_{c0 < j <= t}
// Abar_j and Sc = sum_t e_t Pc(t) over the chunk [c0, c1]:
//   window (Pi, R from (1, 0), the block start's Abar left out): (a0 Pc(c1), a0 Sc), a0 =
//   Abar_c0, or 1 where the chunk starts a block  -> aggX, aggY;
//   reverse (Q, mu_c0 from mu_c1 = 0; the reverse pass's aggregate): (Pc(c1) Abar_{c1+1}, Sc),
//   Abar_{c1+1} = 0 past the sequence end  -> revX, revY.
template <int NS, int MODE>
__global__ void __launch_bounds__(SEL_THREADS, 3) k_sel_win(const float *__restrict__ z, const float *__restrict__ gy,
                                                        const float *__restrict__ b_dt, const float *__restrict__ A,
                                                        float *__restrict__ aggX, float *__restrict__ aggY,
                                                        float *__restrict__ R, int64_t T, int P, int TT,
                                                        int64_t nchunks, int64_t W, float *__restrict__ revX,
                                                        float *__restrict__ revY) {
    extern __shared__ __align__(16) float sm_sel[];
    constexpr int PC = Geo<NS>::PC, SC = Geo<NS>::SC;
    const Stage<NS> sg = stage_carve<NS>(sm_sel);
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int slice = int(blockIdx.y);
    const Geo<NS> g(slice, P);
    const int ZW = P + 2 * NS;
    const int64_t c0 = c * TT, row0 = b * T + c0;
    const int rows = int(c0 + TT <= T ? TT : T - c0);
    const int pp = g.act ? g.p : 0;
    float A2[SEL_NT], pi[SEL_NT], rr[SEL_NT];
    const int64_t ai = ((b * nchunks + c) * P + pp) * NS + g.n0;
#pragma unroll
    for (int k = 0; k < SEL_NT; ++k) {
        A2[k] = A[pp * NS + g.n0 + k] * LOG2E;
        pi[k] = 1.f;
        rr[k] = 0.f;
    }
    if (MODE == 1 && g.act) {
        ld8g(aggX + ai, pi);
        ld8g(aggY + ai, rr);
    }
    StageRegs<NS> RG;
    stage_load<NS, float, false, true>(RG, z, nullptr, gy, b_dt, P, ZW, row0, 0, rows < SC ? rows : SC, slice * PC);
    for (int r0 = 0; r0 < rows; r0 += SC) {
        const int nr = rows - r0 < SC ? rows - r0 : SC;
        __syncthreads();
        stage_store<NS, false, true>(sg, RG, nr, slice * PC, P);
        __syncthreads();
        if (r0 + SC < rows) {
            const int nn = rows - r0 - SC < SC ? rows - r0 - SC : SC;
            stage_load<NS, float, false, true>(RG, z, nullptr, gy, b_dt, P, ZW, row0, r0 + SC, nn, slice * PC);
        }
        for (int r = 0; r < nr; ++r) {
            const float gv = sg.g[r * PC + g.q];
            if (MODE == 1) {
                if ((c0 + r0 + r) % W != 0) {
                    const float dt = sg.dt[r * PC + g.q];
#pragma unroll
                    for (int k = 0; k < SEL_NT; ++k) pi[k] *= ex2(dt * A2[k]);
                }
            } else if (r0 + r > 0) {   // Pc: the factors after the chunk's first token
                const float dt = sg.dt[r * PC + g.q];
#pragma unroll
                for (int k = 0; k < SEL_NT; ++k) pi[k] *= ex2(dt * A2[k]);
            }
            float Cv[SEL_NT];
            ld8s(sg.C + r * NS + g.n0, Cv);
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) rr[k] = fmaf(pi[k], gv * Cv[k], rr[k]);
            if (MODE == 1 && g.act) st8s(R + ((row0 + r0 + r) * P + pp) * NS + g.n0, rr);
        }
    }
    if (MODE == 0 && g.act) {
        // a0: the chunk's first Abar unless the chunk starts a block; Abar of the token after
        const bool starts = c0 % W == 0, has_next = c0 + rows < T;
        const float dt0 = starts ? 0.f : softplus_f(z[row0 * ZW + pp] + b_dt[pp]);
        const float dtn = has_next ? softplus_f(z[(row0 + rows) * ZW + pp] + b_dt[pp]) : 0.f;
        float wx[SEL_NT], wy[SEL_NT], qx[SEL_NT];
#pragma unroll
        for (int k = 0; k < SEL_NT; ++k) {
            const float a0 = starts ? 1.f : ex2(dt0 * A2[k]);
            wx[k] = a0 * pi[k];
            wy[k] = a0 * rr[k];
            qx[k] = has_next ? pi[k] * ex2(dtn * A2[k]) : 0.f;
        }
        st8v(aggX + ai, wx);
        st8v(aggY + ai, wy);
        st8v(revX + ai, qx);
        st8v(revY + ai, rr);
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
// Butterfly transpose-sum of the 2 SEL_NT shares v[] (dB then dC of the thread's states)
// over the warp's channels: levels over lane bits 4..1 halve the values each time, so every
// lane ends with one value summed over the 16 lanes that share its bit 0; with LP == 1
// (one lane a channel) the lane pairs across bit 0 are added last (lanes l, l ^ 1 agree).
template <int LP>
__device__ __forceinline__ float warp_tsum16(float (&v)[2 * SEL_NT], int lane) {
    // (fixed trip counts, so every index is a compile-time constant and v stays in registers)
#pragma unroll
    for (int lv = 0; lv < 4; ++lv) {
        const int s = 16 >> lv, cnt = 8 >> lv;
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
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
// the share index lane l holds after warp_tsum16
__device__ __forceinline__ int tsum16_index(int lane) {
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Running count of the warps done with a stage: acquire-release, so the last warp's refill
// is ordered after every warp's reads of the stage.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
    return old;
}

constexpr int SEL_NSTG = 3;   // stages in the ring of state rows
template <bool TRUNC>
constexpr int sel_group() { return TRUNC ? 1 : 2; }   // tokens a stage

// MODE 0: chunk aggregates of the reverse scan (Q = prod_{c0 < j <= c1} Abar_j, S = mu_c0
// from mu_c1 = 0) -> aggX, aggY.  256 threads.
// MODE 1: outputs from the carries (q_in, mu_in) in aggX, aggY: dz[:, :P] (the dt part,
// through the softplus), the CTA's partial sums over its channels of dB and dC per token
// -> bc [B*T, nslices, 2 NS], and the chunk's dA partial -> dAp [B*nchunks, P, NS].
// TRUNC: mu^W = mu + q R(min(t+W-1, T-1)) where a later block exists and t starts none.
// The state rows (and R rows) arrive by bulk copies into a ring of stages: stage k holds the
// rows of group k (tokens counted down from the chunk's top, G a group), one more stage the
// row before the chunk; group k reads stages k and k + 1.  Thread 0 issues the first stages;
// afterwards the last of the eight warps to finish with a stage refills it, so no thread
// waits for a stage to drain and the 8 warps keep 128 registers a thread.
// INP (MODE 1, stacked layers): also the input path's share that does not go through the
// projection, dxd = dt sum_n mu^W B (xhat's factor in the input term), written as
// gadd = gy + dxd / r (r: the rms of the layer's input stream), and the CTA's partial row
// dots xhat . dxhat = sum_p (dz_dt,p z_p + xhat_p dxd_p) -> rowdot [B*T, nslices + 1]
// (the last slice is k_sel_bc_reduce's, for the dB and dC columns; together with dz z they
// give xhat . (dz W_in^T) without the product, since z = xhat W_in).
template <int NS, typename TX, typename TD, int MODE, bool TRUNC, bool INP = false>
__global__ void __launch_bounds__(SEL_THREADS, 2) k_sel_bwd(const float *__restrict__ z, const TX *__restrict__ x,
                                                            const float *__restrict__ gy, const float *__restrict__ h,
                                                            const float *__restrict__ R, const float *__restrict__ b_dt,
                                                            const float *__restrict__ A, float *__restrict__ aggX,
                                                            float *__restrict__ aggY, TD *__restrict__ dz,
                                                            float *__restrict__ bc, float *__restrict__ dAp, int64_t T,
                                                            int P, int TT, int64_t nchunks, int nslices, int64_t W,
                                                            unsigned *status, const float *__restrict__ rin,
                                                            float *__restrict__ gadd, float *__restrict__ rowdot) {
    extern __shared__ __align__(16) float sm_sel[];
    constexpr int PC = Geo<NS>::PC, LP = Geo<NS>::LP, SC = Geo<NS>::SC;
    constexpr int G = sel_group<TRUNC>();
    constexpr int RF = PC * NS;                            // floats of one row segment
    constexpr int STG = G * RF * (TRUNC ? 2 : 1);          // floats a stage
    __shared__ uint64_t s_full[SEL_NSTG];
    __shared__ unsigned s_done[SEL_NSTG];                  // warps done with each slot, running
    __shared__ int s_abort;
    __shared__ float s_rd[SEL_THREADS / 32][16];           // INP: the warps' row-dot shares
    __shared__ float s_rin[16];                            // INP: the sub-chunk's 1 / r
    const Stage<NS> sg = stage_carve<NS>(sm_sel, INP);
    float *sW = sm_sel + stage_floats<NS>(INP);            // [8 warps][SC][32]
    float *sH = sW + (SEL_THREADS / 32) * SC * 32;         // [SEL_NSTG][STG]
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int slice = int(blockIdx.y);
    const int ZW = P + 2 * NS, lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    const int64_t c0 = c * TT, row0 = b * T + c0;
    const int rows = int(c0 + TT <= T ? TT : T - c0);
    const int p0 = slice * PC;
    const int ngroups = (rows + G - 1) / G;
    const int nst = ngroups + (c0 > 0 ? 1 : 0);

    // the bulk copies of stage k (one thread): the rows of group k, or the row before the chunk
    auto issue_stage = [&](int k) {
        const int pw = P - p0 < PC ? P - p0 : PC;
        const uint32_t rowb = uint32_t(pw) * NS * 4u;
        const int slot = k % SEL_NSTG;
        const uint32_t bar = smem_u32(&s_full[slot]);
        float *dst = sH + slot * STG;
        if (k < ngroups) {
            const int hi = rows - G * k, lo = hi - G > 0 ? hi - G : 0, n = hi - lo;
            mbar_arrive_expect_tx(bar, uint32_t(n) * rowb * (TRUNC ? 2u : 1u));
            for (int j = 0; j < n; ++j)
                bulk_g2s(smem_u32(dst + j * RF), h + ((row0 + lo + j) * P + p0) * NS, rowb, bar);
            if (TRUNC)
                for (int j = 0; j < n; ++j) {
                    const int64_t t = c0 + lo + j, m = t + W - 1 < T - 1 ? t + W - 1 : T - 1;
                    bulk_g2s(smem_u32(dst + (G + j) * RF), R + ((b * T + m) * P + p0) * NS, rowb, bar);
                }
        } else {
            mbar_arrive_expect_tx(bar, rowb);
            bulk_g2s(smem_u32(dst), h + ((row0 - 1) * P + p0) * NS, rowb, bar);
        }
    };
    if (MODE == 1) {
        if (threadIdx.x == 0) {
            for (int j = 0; j < SEL_NSTG; ++j) {
                mbar_init(smem_u32(&s_full[j]), 1);
                s_done[j] = 0u;
            }
            s_abort = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (threadIdx.x == 0)
            for (int k = 0; k < nst && k < SEL_NSTG; ++k) issue_stage(k);
    }

    const Geo<NS> g(slice, P);
    const int pp = g.act ? g.p : 0;   // lanes past P walk on zeros (the lane sums need them)
    float A2[SEL_NT], mu[SEL_NT], qv[SEL_NT], abn[SEL_NT], dA[SEL_NT], hc[SEL_NT];
    const int64_t ai = ((b * nchunks + c) * P + pp) * NS + g.n0;
    const bool has_next = c0 + rows < T;
    const float dtn = has_next ? softplus_f(z[(row0 + rows) * ZW + pp] + b_dt[pp]) : 0.f;
#pragma unroll
    for (int k = 0; k < SEL_NT; ++k) {
        A2[k] = A[pp * NS + g.n0 + k] * LOG2E;
        abn[k] = has_next ? ex2(dtn * A2[k]) : 0.f;   // Abar of the token after the chunk
        mu[k] = 0.f;
        qv[k] = 1.f;
        dA[k] = 0.f;
        hc[k] = 0.f;
    }
    if (MODE == 1 && g.act) {
        ld8g(aggY + ai, mu);
        if (TRUNC) ld8g(aggX + ai, qv);
    }
    const bool next_block = TRUNC && (c0 / W + 1) * W < T;
    const int off = g.q * NS + g.n0;

    // flush the warp sums of the tokens [lo_s, hi_s) of the last sub-chunk to bc
    auto flush = [&](int lo_s, int hi_s) {
        for (int e = threadIdx.x; e < SC * 32; e += SEL_THREADS) {
            const int j = e / 32, l = e % 32;
            if (j >= hi_s - lo_s || (LP == 1 && (l & 1))) continue;
            float acc = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < SEL_THREADS / 32; ++w8) acc += sW[(w8 * SC + j) * 32 + l];
            const int vi = tsum16_index(l), which = vi >> 3;
            const int n = (LP == 2 ? (l & 1) : 0) * SEL_NT + (vi & 7);
            const int64_t trow = row0 + (hi_s - 1 - j);
            bc[(trow * nslices + slice) * (2 * NS) + which * NS + n] = acc;
        }
        if (INP)
            for (int j = threadIdx.x; j < hi_s - lo_s; j += SEL_THREADS) {
                float acc = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < SEL_THREADS / 32; ++w8) acc += s_rd[w8][j];
                rowdot[(row0 + (hi_s - 1 - j)) * (nslices + 1) + slice] = acc;
            }
        // dz's dt columns (from the sigma slots) and gadd (from the z slots) of the sub-chunk's
        // rows [lo_s, hi_s), 8 channels a thread-step (P is a multiple of 8)
        const int pw = P - p0 < PC ? P - p0 : PC;
        for (int e = threadIdx.x; e < (hi_s - lo_s) * (PC / 8); e += SEL_THREADS) {
            const int j = e / (PC / 8), c8 = (e % (PC / 8)) * 8;
            if (c8 >= pw) continue;
            const int64_t trow = row0 + lo_s + j;
            const float4 a0 = *reinterpret_cast<const float4 *>(sg.sig + j * PC + c8);
            const float4 a1 = *reinterpret_cast<const float4 *>(sg.sig + j * PC + c8 + 4);
            TD *dst = dz + trow * ZW + p0 + c8;
            if constexpr (sizeof(TD) == 2) {
                uint4 u;
                u.x = pack_bf16x2(a0.x, a0.y);
                u.y = pack_bf16x2(a0.z, a0.w);
                u.z = pack_bf16x2(a1.x, a1.y);
                u.w = pack_bf16x2(a1.z, a1.w);
                *reinterpret_cast<uint4 *>(dst) = u;
            } else {
                reinterpret_cast<float4 *>(dst)[0] = a0;
                reinterpret_cast<float4 *>(dst)[1] = a1;
            }
            if (INP) {
                float *gdst = gadd + trow * P + p0 + c8;
                reinterpret_cast<float4 *>(gdst)[0] = *reinterpret_cast<const float4 *>(sg.zr + j * PC + c8);
                reinterpret_cast<float4 *>(gdst)[1] = *reinterpret_cast<const float4 *>(sg.zr + j * PC + c8 + 4);
            }
        }
    };

    int slo = rows, shi = rows;   // the staged sub-chunk [slo, shi)
    StageRegs<NS> R0;             // MODE 0: the next sub-chunk's inputs
    for (int gi = 0; gi < ngroups; ++gi) {
        const int hi = rows - G * gi, lo = hi - G > 0 ? hi - G : 0;
        if (hi == slo || gi == 0) {   // a new sub-chunk of the per-token inputs
            walkers_sync();
            if (MODE == 1 && gi > 0) {
                flush(slo, shi);
                walkers_sync();
            }
            shi = hi;
            slo = hi - SC > 0 ? hi - SC : 0;
            if (MODE == 0) {   // registers to spare: the next sub-chunk loads while this one is walked
                if (gi == 0) stage_load<NS, TX, false, true>(R0, z, x, gy, b_dt, P, ZW, row0, slo, shi - slo, p0);
                stage_store<NS, false, true>(sg, R0, shi - slo, p0, P);
                if (slo > 0) {
                    const int nlo = slo - SC > 0 ? slo - SC : 0;
                    stage_load<NS, TX, false, true>(R0, z, x, gy, b_dt, P, ZW, row0, nlo, slo - nlo, p0);
                }
            } else {
                stage_sub<NS, TX, true, true, INP>(sg, z, x, gy, b_dt, P, ZW, row0, slo, shi - slo, p0);
                if (INP)
                    for (int j = threadIdx.x; j < shi - slo; j += SEL_THREADS)
                        s_rin[j] = 1.f / __ldg(rin + row0 + slo + j);
                // the next sub-chunk's inputs into L2 while this one is walked
                if (slo > 0) {
                    const int nlo = slo - SC > 0 ? slo - SC : 0;
                    stage_prefetch<NS, TX>(z, x, gy, P, ZW, row0, nlo, slo - nlo, p0);
                }
            }
            walkers_sync();
        }
        const float *stg = sH + (gi % SEL_NSTG) * STG;
        if (MODE == 1) {
            mbar_wait(smem_u32(&s_full[gi % SEL_NSTG]), uint32_t((gi / SEL_NSTG) & 1), &s_abort, status);
            if (gi == 0 && g.act) ld8s(stg + (hi - 1 - lo) * RF + off, hc);   // h of the chunk's last token
            if (gi + 1 < nst)
                mbar_wait(smem_u32(&s_full[(gi + 1) % SEL_NSTG]), uint32_t(((gi + 1) / SEL_NSTG) & 1), &s_abort,
                          status);
        }
        for (int r = hi - 1; r >= lo; --r) {
            const int rr = r - slo;
            const float gv = sg.g[rr * PC + g.q], dt = sg.dt[rr * PC + g.q];
            float Cv[SEL_NT], ab[SEL_NT];
            ld8s(sg.C + rr * NS + g.n0, Cv);
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) {
                mu[k] = fmaf(abn[k], mu[k], gv * Cv[k]);
                if (MODE == 0 || TRUNC) qv[k] *= abn[k];
                ab[k] = ex2(dt * A2[k]);
            }
            if (MODE == 1) {
                // h_{r-1}: the row below in this stage, the top row of the next stage, or zero
                float hp[SEL_NT], Bv[SEL_NT], v[2 * SEL_NT];
#pragma unroll
                for (int k = 0; k < SEL_NT; ++k) hp[k] = 0.f;
                if (g.act) {
                    if (r > lo) ld8s(stg + (r - 1 - lo) * RF + off, hp);
                    else if (gi + 1 < nst) {
                        const int lo2 = lo - G > 0 ? lo - G : 0;
                        const int top = gi + 1 < ngroups ? lo - 1 - lo2 : 0;
                        ld8s(sH + ((gi + 1) % SEL_NSTG) * STG + top * RF + off, hp);
                    }
                }
                float mw[SEL_NT];   // the window sum mu^W of this token (the scan keeps mu)
#pragma unroll
                for (int k = 0; k < SEL_NT; ++k) mw[k] = mu[k];
                if (TRUNC && next_block && (c0 + r) % W != 0 && g.act) {
                    float rv[SEL_NT];
                    ld8s(stg + (G + r - lo) * RF + off, rv);
#pragma unroll
                    for (int k = 0; k < SEL_NT; ++k) mw[k] = fmaf(qv[k], rv[k], mu[k]);
                }
                ld8s(sg.B + rr * NS + g.n0, Bv);
                const float xv = sg.x[rr * PC + g.q], dtx = dt * xv;
                float dda = 0.f, ddb = 0.f;
#pragma unroll
                for (int k = 0; k < SEL_NT; ++k) {
                    const float ma = mw[k] * (ab[k] * hp[k]);
                    dda = fmaf(A2[k], ma, dda);
                    ddb = fmaf(mw[k], Bv[k], ddb);
                    dA[k] = fmaf(dt, ma, dA[k]);
                    v[k] = mw[k] * dtx;             // dB_t,n share
                    v[SEL_NT + k] = gv * hc[k];     // dC_t,n share
                    hc[k] = hp[k];
                }
                const float ddt = chan_sum<LP>(fmaf(dda, 1.f / LOG2E, ddb * xv));
                // dz's dt column (through the softplus) replaces sigma in its shared slot and
                // goes out with the sub-chunk's flush, as whole rows
                float dzs = 0.f;   // dz_dt as stored
                if (g.act && g.n0 == 0) {
                    const float val = ddt * sg.sig[rr * PC + g.q];
                    sg.sig[rr * PC + g.q] = val;
                    if constexpr (sizeof(TD) == 2) dzs = __bfloat162float(__float2bfloat16_rn(val));
                    else dzs = val;
                }
                if (INP) {
                    const float dxd = dt * chan_sum<LP>(ddb);
                    float rd = 0.f;
                    if (g.act && g.n0 == 0) {
                        rd = fmaf(dzs, sg.zr[rr * PC + g.q], xv * dxd);
                        sg.zr[rr * PC + g.q] = sg.g[rr * PC + g.q] + dxd * s_rin[rr];   // gadd, flushed too
                    }
                    // a channel's value sits on its first lane: with two lanes a channel the odd
                    // lanes hold zeros and the last level is not needed
#pragma unroll
                    for (int o = 16; o >= (LP == 2 ? 2 : 1); o >>= 1) rd += __shfl_xor_sync(0xffffffffu, rd, o);
                    if (lane == 0) s_rd[wp][shi - 1 - r] = rd;
                }
                sW[(wp * SC + (shi - 1 - r)) * 32 + lane] = warp_tsum16<LP>(v, lane);
            }
#pragma unroll
            for (int k = 0; k < SEL_NT; ++k) abn[k] = ab[k];
        }
        if (MODE == 1) {
            __syncwarp();   // the warp's reads of the stage are done
            if (lane == 0) {
                const int slot = gi % SEL_NSTG;
                const unsigned prev = atom_add_acq_rel(&s_done[slot], 1u);
                if (prev % (SEL_THREADS / 32) == SEL_THREADS / 32 - 1 && gi + SEL_NSTG < nst) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // reads before the copies' writes
                    issue_stage(gi + SEL_NSTG);
                }
            }
        }
    }
    if (MODE == 1) {
        walkers_sync();
        flush(slo, shi);
    }
    if (!g.act) return;
    if (MODE == 0) {
        st8v(aggX + ai, qv);
        st8v(aggY + ai, mu);
    } else {
        st8v(dAp + ((b * nchunks + c) * P + g.p) * NS + g.n0, dA);
    }
}

// dz[:, P + j] = sum over slices of bc (j < 2 NS), in the dz storage type.  With rowdot
// (stacked layers): the row's sum_j dz_P+j z_P+j (as stored) -> rowdot[r * (nslices + 1) + nslices];
// a row's NS2 threads are adjacent lanes (NS2 = 16 or 32).
template <typename TD>
__global__ void k_sel_bc_reduce(const float *__restrict__ bc, TD *__restrict__ dz, int64_t rows, int P, int NS2,
                                int nslices, const float *__restrict__ z, float *__restrict__ rowdot) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool live = i < rows * NS2;
    const int64_t r = i / NS2;
    const int j = int(i % NS2);
    float sv = 0.f;
    if (live) {
        float acc = 0.f;
        for (int s = 0; s < nslices; ++s) acc += bc[(r * nslices + s) * NS2 + j];
        if constexpr (sizeof(TD) == 2) {
            const __nv_bfloat16 vb = __float2bfloat16_rn(acc);
            dz[r * (P + NS2) + P + j] = vb;
            sv = __bfloat162float(vb);
        } else {
            dz[r * (P + NS2) + P + j] = acc;
            sv = acc;
        }
    }
    if (rowdot == nullptr) return;
    float c = live ? sv * z[r * (P + NS2) + P + j] : 0.f;
    for (int o = NS2 / 2; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o, NS2);
    if (live && j == 0) rowdot[r * (nslices + 1) + nslices] = c;
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
                             const float *xres, float *aggX, float *aggY, int64_t B, int64_t T, int P, cudaStream_t st) {
    const int TT = sel_chunk(T, 0);
    const int64_t nchunks = (T + TT - 1) / TT;
    const dim3 grid = sel_grid(B, nchunks, P, NS);
    const size_t smem = stage_floats<NS>() * 4;
    const TX *xt = static_cast<const TX *>(x);
    cudaError_t e;
    if ((e = smem_attr(k_sel_fwd<NS, TX, 0>, smem)) != cudaSuccess) return e;
    if ((e = smem_attr(k_sel_fwd<NS, TX, 1>, smem)) != cudaSuccess) return e;
    if ((e = smem_attr(k_sel_fwd<NS, TX, 1, true>, smem)) != cudaSuccess) return e;
    k_sel_fwd<NS, TX, 0><<<grid, SEL_THREADS, smem, st>>>(z, xt, b_dt, A, aggX, aggY, h, y, nullptr, T, P, TT,
                                                          nchunks);
    const int64_t n = B * int64_t(P) * NS;
    k_sel_carry<0><<<unsigned((n + 255) / 256), 256, 0, st>>>(aggX, aggY, B, int64_t(P) * NS, nchunks, T, TT, T);
    if (xres)
        k_sel_fwd<NS, TX, 1, true><<<grid, SEL_THREADS, smem, st>>>(z, xt, b_dt, A, aggX, aggY, h, y, xres, T, P, TT,
                                                                    nchunks);
    else
        k_sel_fwd<NS, TX, 1><<<grid, SEL_THREADS, smem, st>>>(z, xt, b_dt, A, aggX, aggY, h, y, nullptr, T, P, TT,
                                                              nchunks);
    return cudaGetLastError();
}

cudaError_t launch_sel_fwd(const float *z, const void *x, bool x_bf16, const float *b_dt, const float *A, float *h,
                           float *y, const float *xres, float *aggX, float *aggY, int64_t B, int64_t T, int P, int NS,
                           cudaStream_t st) {
    if (NS == 16) return x_bf16 ? sel_fwd_t<16, __nv_bfloat16>(z, x, b_dt, A, h, y, xres, aggX, aggY, B, T, P, st)
                                : sel_fwd_t<16, float>(z, x, b_dt, A, h, y, xres, aggX, aggY, B, T, P, st);
    if (NS == 8) return x_bf16 ? sel_fwd_t<8, __nv_bfloat16>(z, x, b_dt, A, h, y, xres, aggX, aggY, B, T, P, st)
                               : sel_fwd_t<8, float>(z, x, b_dt, A, h, y, xres, aggX, aggY, B, T, P, st);
    return cudaErrorInvalidValue;
}

template <int NS, typename TX, typename TD>
static cudaError_t sel_bwd_t(const float *z, const void *x, const float *gy, const float *h, const float *b_dt,
                             const float *A, void *dz, float *dA, const SelBwdWs &w, const SelInp &inp, int64_t B,
                             int64_t T, int P, int64_t W, unsigned *status, cudaStream_t st) {
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
        const size_t sm1 = stage_floats<NS>() * 4;
        if ((e = smem_attr(k_sel_win<NS, 0>, sm1)) != cudaSuccess) return e;
        if ((e = smem_attr(k_sel_win<NS, 1>, sm1)) != cudaSuccess) return e;
        // one walk gives both scans' chunk aggregates (the reverse ones into aggX, aggY)
        k_sel_win<NS, 0><<<grid, SEL_THREADS, sm1, st>>>(z, gy, b_dt, A, w.winX, w.winY, w.R, T, P, TT, nchunks, Wk,
                                                         w.aggX, w.aggY);
        k_sel_carry<2><<<cgrid, 256, 0, st>>>(w.winX, w.winY, B, int64_t(P) * NS, nchunks, T, TT, Wk);
        k_sel_win<NS, 1><<<grid, SEL_THREADS, sm1, st>>>(z, gy, b_dt, A, w.winX, w.winY, w.R, T, P, TT, nchunks, Wk,
                                                         nullptr, nullptr);
    }
    // MODE 0: the staged inputs; MODE 1: also the warp sums and the ring of row stages (and,
    // with the input path, the raw z of the dt columns)
    const bool inpath = inp.gadd != nullptr;
    const size_t sm0 = stage_floats<NS>() * 4;
    const size_t sm_ws = size_t(SEL_THREADS / 32) * Geo<NS>::SC * 32 * 4;
    const size_t row_seg = size_t(Geo<NS>::PC) * NS * 4;
#define ADJ_SEL_BWD(TR, IN)                                                                                        \
    do {                                                                                                           \
        const size_t sm1 = stage_floats<NS>(IN) * 4 + sm_ws +                                                      \
                           size_t(SEL_NSTG) * sel_group<TR>() * row_seg * (TR ? 2 : 1);                            \
        if ((e = smem_attr(k_sel_bwd<NS, TX, TD, 1, TR, IN>, sm1)) != cudaSuccess) return e;                       \
        if (!TR) { /* the truncated form has its reverse aggregates from the window walk */                        \
            if ((e = smem_attr(k_sel_bwd<NS, TX, TD, 0, TR>, sm0)) != cudaSuccess) return e;                       \
            k_sel_bwd<NS, TX, TD, 0, TR><<<grid, SEL_THREADS, sm0, st>>>(z, xt, gy, h, w.R, b_dt, A, w.aggX,       \
                                                                         w.aggY, dzt, w.bc, w.dAp, T, P, TT,       \
                                                                         nchunks, nsl, Wk, status, nullptr,        \
                                                                         nullptr, nullptr);                        \
        }                                                                                                          \
        k_sel_carry<1><<<cgrid, 256, 0, st>>>(w.aggX, w.aggY, B, int64_t(P) * NS, nchunks, T, TT, Wk);             \
        k_sel_bwd<NS, TX, TD, 1, TR, IN><<<grid, SEL_THREADS, sm1, st>>>(                                      \
            z, xt, gy, h, w.R, b_dt, A, w.aggX, w.aggY, dzt, w.bc, w.dAp, T, P, TT, nchunks, nsl, Wk, status,      \
            inp.r, inp.gadd, inp.rowdot);                                                                          \
    } while (0)
    if (trunc) {
        if (inpath) ADJ_SEL_BWD(true, true);
        else ADJ_SEL_BWD(true, false);
    } else {
        if (inpath) ADJ_SEL_BWD(false, true);
        else ADJ_SEL_BWD(false, false);
    }
#undef ADJ_SEL_BWD
    const int64_t nbc = B * T * 2 * NS;
    k_sel_bc_reduce<TD><<<unsigned((nbc + 255) / 256), 256, 0, st>>>(w.bc, dzt, B * T, P, 2 * NS, nsl,
                                                                     inpath ? z : nullptr, inp.rowdot);
    k_sel_rows_sum<<<unsigned((int64_t(P) * NS + 255) / 256), 256, 0, st>>>(w.dAp, dA, B * nchunks,
                                                                          int64_t(P) * NS);
    return cudaGetLastError();
}

cudaError_t launch_sel_bwd(const float *z, const void *x, bool x_bf16, const float *gy, const float *h,
                           const float *b_dt, const float *A, void *dz, bool d_bf16, float *dA, const SelBwdWs &w,
                           const SelInp &inp, int64_t B, int64_t T, int P, int NS, int64_t W, unsigned *status,
                           cudaStream_t st) {
#define ADJ_SEL_B(NSV)                                                                                              \
    do {                                                                                                            \
        if (x_bf16) {                                                                                               \
            if (d_bf16)                                                                                             \
                return sel_bwd_t<NSV, __nv_bfloat16, __nv_bfloat16>(z, x, gy, h, b_dt, A, dz, dA, w, inp, B, T, P,  \
                                                                    W, status, st);                                 \
            return sel_bwd_t<NSV, __nv_bfloat16, float>(z, x, gy, h, b_dt, A, dz, dA, w, inp, B, T, P, W, status,  \
                                                        st);                                                        \
        }                                                                                                           \
        if (d_bf16)                                                                                                 \
            return sel_bwd_t<NSV, float, __nv_bfloat16>(z, x, gy, h, b_dt, A, dz, dA, w, inp, B, T, P, W, status,  \
                                                        st);                                                        \
        return sel_bwd_t<NSV, float, float>(z, x, gy, h, b_dt, A, dz, dA, w, inp, B, T, P, W, status, st);          \
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
