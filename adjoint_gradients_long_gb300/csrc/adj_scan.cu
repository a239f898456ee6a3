// adj_scan.cu -- single-pass chunked scans with decoupled look-back for the diagonal
// linear recurrences of the adjoint-sharding path.
//
// Source: the review page "Adjoint sharding for very long context training of state
// space models" ([AS]).
//   * forward state scan   h_t = a_t h_{t-1} + u_t                 ([AS] Assumptions, Sec. 3.1)
//   * reverse adjoint scan mu_i = g_i c_i + a_{i+1} mu_{i+1}: the sum over t of
//     dl_t/dy_t lambda_{t,i}, lambda_{t,i} = C_t prod_{j=i+1..t} A_j, computed backwards
//     as in [AS] What carries the argument (Proposition 1) and Figure 4
//   * truncated adjoint   mu^W_i = sum_{t=i}^{min(T-1,i+W-1)} g_t c_t prod_{j=i+1..t} a_j
//     ([AS] Core claim, truncated adjoint sharding), evaluated blockwise without
//     subtraction: with blocks of W tokens and s the start of the block after i's,
//        mu^W_i = S_i + Q_i R(i+W-1),
//        S_i = sum_{t=i}^{s-1} e_t prod_{j=i+1..t} a_j,  Q_i = prod_{j=i+1..s} a_j,
//        R(m) = sum_{t=s}^{m} e_t prod_{j=s+1..t} a_j  (R(s-1) = 0),  e = g c.
//     (S_i, Q_i) is the reverse scan restarted at every block end; R is a forward
//     scan restarted at every block start (k_win_scan).  Every product spans at most
//     W factors.
//
// Work decomposition (all three kernels): a CTA of 8 warps owns one chunk of
// 8*L consecutive tokens of one sequence and 128 channels (lane = 4 channels, one
// float4 per token row, so every warp access is a 512-byte coalesced row segment).
// Warp w owns tokens [chunk*8L + w*L, +L).  Each thread reduces its L tokens to one
// composite map, the 8 warp composites are combined in shared memory, and warp 0
// publishes the chunk aggregate and looks back over its predecessors' descriptors
// (decoupled look-back).  Chunks are numbered by an atomic ticket in scan order,
// so a CTA only ever waits for CTAs that started before it; every wait is bounded.
#include "adj_internal.cuh"

namespace adj {

constexpr int SC_WARPS = 8;
constexpr int SC_LB_BATCH = 2;       // descriptor loads in flight per look-back batch
constexpr int SC_SLICE = 128;        // channels per CTA
constexpr int SC_MIN_CHUNK = 32;     // smallest chunk (L = 4); sizes the descriptor arrays
constexpr unsigned F_AGG = 1u, F_INC = 2u;

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
static inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

size_t scan_ws_bytes(int64_t B, int64_t T, int N) {
    int64_t n = B * cdiv(N, SC_SLICE) * cdiv(T, SC_MIN_CHUNK);
    return 256 + al256(size_t(n) * 4) + 4 * al256(size_t(n) * 32 * sizeof(float4));
}

ScanWs scan_ws_carve(void *base, int64_t B, int64_t T, int N) {
    int64_t n = B * cdiv(N, SC_SLICE) * cdiv(T, SC_MIN_CHUNK);
    char *p = static_cast<char *>(base);
    ScanWs d;
    d.ticket = reinterpret_cast<unsigned *>(p);
    p += 256;
    d.flags = reinterpret_cast<unsigned *>(p);
    p += al256(size_t(n) * 4);
    size_t db = al256(size_t(n) * 32 * sizeof(float4));
    d.agg0 = reinterpret_cast<float4 *>(p); p += db;
    d.agg1 = reinterpret_cast<float4 *>(p); p += db;
    d.inc0 = reinterpret_cast<float4 *>(p); p += db;
    d.inc1 = reinterpret_cast<float4 *>(p);
    return d;
}

// bytes of the ticket + flags prefix that must be zero before a launch
static size_t scan_reset_bytes(int64_t B, int64_t T, int N) {
    int64_t n = B * cdiv(N, SC_SLICE) * cdiv(T, SC_MIN_CHUNK);
    return 256 + al256(size_t(n) * 4);
}

// Publish one or two float4 per lane and then the flag (release after a fence).
__device__ __forceinline__ void warp_publish(float4 *p0, float4 v0, float4 *p1, float4 v1,
                                             unsigned *flag, unsigned fval, int lane) {
    if (p0) st_cg4(p0, v0);
    if (p1) st_cg4(p1, v1);
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(flag, fval);
}


// Warp-wide decoupled look-back.  The predecessors of a chunk, nearest first, are
// p0, p0 + dir, p0 + 2 dir, ... (count of them).  Each round, lane i reads the flag of
// the i-th not yet consumed predecessor; the warp then folds, for its own channels,
// every published aggregate up to the nearest inclusive prefix (or up to the first
// predecessor that has published nothing yet, which it then waits for).  Descriptor
// loads of one round are issued in batches, so a round costs about two L2 round trips
// however many predecessors it folds.  extend(acc, agg) folds one more aggregate;
// finish(acc, inc) returns the carry.  A wait that gives up finishes with `zero_inc`.
template <class C, class LA, class LI, class EX, class FI>
__device__ __forceinline__ C warp_lookback(const unsigned *flags, int64_t p0, int dir, int64_t count, C acc,
                                           LA load_agg, LI load_inc, EX extend, FI finish, C zero_inc,
                                           unsigned *status, int lane) {
    int64_t done = 0;
    for (int round = 0; round < SPIN_LIMIT; ++round) {
        const bool exists = done + lane < count;
        const unsigned f = exists ? ld_acquire(&flags[p0 + dir * (done + lane)]) : 0u;
        const unsigned incl = __ballot_sync(0xffffffffu, exists && f == F_INC);
        const unsigned miss = __ballot_sync(0xffffffffu, exists && f == 0u);
        __syncwarp();   // orders every lane's descriptor loads after the flag acquires above
        const int ji = incl ? __ffs(int(incl)) - 1 : 32, jm = miss ? __ffs(int(miss)) - 1 : 32;
        int m = ji < jm ? ji : jm;
        if (int64_t(m) > count - done) m = int(count - done);
        for (int i0 = 0; i0 < m; i0 += SC_LB_BATCH) {
            C t[SC_LB_BATCH];
#pragma unroll
            for (int b = 0; b < SC_LB_BATCH; ++b)
                if (i0 + b < m) t[b] = load_agg(p0 + dir * (done + i0 + b));
#pragma unroll
            for (int b = 0; b < SC_LB_BATCH; ++b)
                if (i0 + b < m) acc = extend(acc, t[b]);
        }
        done += m;
        if (ji < jm && ji == m) return finish(acc, load_inc(p0 + dir * done));
        if (done >= count) return finish(acc, zero_inc);   // not reached: the first chunk is always inclusive
        if (m == 0) {
            // the nearest predecessor has published nothing yet: wait for it
            unsigned fw = 0;
            if (lane == 0) fw = wait_flag(&flags[p0 + dir * done], status);
            fw = __shfl_sync(0xffffffffu, fw, 0);
            if (fw == 0) return finish(acc, zero_inc);
        }
    }
    record_timeout(status);
    return finish(acc, zero_inc);
}

// ============================================================================ forward state scan
// Composite of a token range: h_out = A h_in + H.  (A2,H2) after (A1,H1) = (A2 A1, A2 H1 + H2).
struct float2x4 {
    float4 x, y;
};
template <int L, int LB>
__global__ void __launch_bounds__(256, 3) k_fwd_scan(const float *__restrict__ a, const float *__restrict__ u,
                                                  float *__restrict__ h, int64_t T, int N, int nslices,
                                                  int64_t nseq, int64_t nchunks, ScanWs d, unsigned *status) {
    __shared__ unsigned s_ticket;
    __shared__ float4 sA[SC_WARPS][32], sH[SC_WARPS][32], sC[32];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) s_ticket = atomicAdd(d.ticket, 1u);
    __syncthreads();
    const int64_t tk = s_ticket, chunk = tk / nseq, seq = tk % nseq;
    const int64_t b = seq / nslices;
    const int ch = int(seq % nslices) * SC_SLICE + lane * 4;
    const bool act = ch < N;
    const int64_t t0 = chunk * (SC_WARPS * L) + w * L;
    const int64_t base = b * T * N + ch;

    // pass 1: only the composite of this thread's L tokens is kept (folded LB rows at a
    // time); the rows stay in L2 and are read again in pass 2, so few registers are
    // live across the look-back and three CTAs fit per SM.
    float4 A = f4(1.f), H = f4(0.f);
    for (int k0 = 0; k0 < L; k0 += LB) {
        float4 av[LB], uv[LB];
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            const int64_t t = t0 + k0 + k;
            const bool ok = act && t < T;
            av[k] = ok ? ld_l2keep4(a + base + t * N) : f4(1.f);
            uv[k] = ok ? ld_l2keep4(u + base + t * N) : f4(0.f);
        }
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            H = fma4(av[k], H, uv[k]);
            A = A * av[k];
        }
    }
    sA[w][lane] = A;
    sH[w][lane] = H;
    __syncthreads();

    if (w == 0) {
        float4 cA = f4(1.f), cH = f4(0.f);
#pragma unroll
        for (int j = 0; j < SC_WARPS; ++j) {
            cH = fma4(sA[j][lane], cH, sH[j][lane]);
            cA = cA * sA[j][lane];
        }
        const int64_t di = seq * nchunks + chunk;
        float4 carry = f4(0.f);
        if (chunk > 0) {
            warp_publish(&d.agg0[di * 32 + lane], cA, &d.agg1[di * 32 + lane], cH, &d.flags[di], F_AGG, lane);
            const int64_t fb = seq * nchunks;
            // acc = composite of the chunks between the inclusive prefix found and this chunk
            const float2x4 r = warp_lookback<float2x4>(
                d.flags + fb, chunk - 1, -1, chunk, float2x4{f4(1.f), f4(0.f)},
                [&](int64_t p) { return float2x4{ld_cg4(&d.agg0[(fb + p) * 32 + lane]), ld_cg4(&d.agg1[(fb + p) * 32 + lane])}; },
                [&](int64_t p) { return float2x4{f4(0.f), ld_cg4(&d.inc1[(fb + p) * 32 + lane])}; },
                [](const float2x4 &acc, const float2x4 &g) { return float2x4{acc.x * g.x, fma4(acc.x, g.y, acc.y)}; },
                [](const float2x4 &acc, const float2x4 &inc) { return float2x4{f4(0.f), fma4(acc.x, inc.y, acc.y)}; },
                float2x4{f4(0.f), f4(0.f)}, status, lane);
            carry = r.y;
        }
        warp_publish(nullptr, f4(0.f), &d.inc1[di * 32 + lane], fma4(cA, carry, cH), &d.flags[di], F_INC, lane);
        sC[lane] = carry;
    }
    __syncthreads();

    float4 hc = sC[lane];
    for (int j = 0; j < w; ++j) hc = fma4(sA[j][lane], hc, sH[j][lane]);
    for (int k0 = 0; k0 < L; k0 += LB) {
        float4 av[LB], uv[LB];
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            const int64_t t = t0 + k0 + k;
            const bool ok = act && t < T;
            av[k] = ok ? ld_stream4(a + base + t * N) : f4(1.f);
            uv[k] = ok ? ld_stream4(u + base + t * N) : f4(0.f);
        }
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            hc = fma4(av[k], hc, uv[k]);
            const int64_t t = t0 + k0 + k;
            if (act && t < T) st_stream4(h + base + t * N, hc);
        }
    }
}

// ============================================================================ window scan R
// Forward scan restarted at every multiple of W.  Token m maps the state (P, R) to
// (a_m P, R + e_m a_m P); a block-start token resets it to (1, e_m).  Composite of a
// range: (Pi, Sig, closed); Y after X = Y.closed ? Y : (X.Pi Y.Pi, X.Sig + X.Pi Y.Sig, X.closed).
// Output R_m = Sig of the composite from the block start to m.
struct FwdSeg {
    float4 P, S;
    bool cl;
};
__device__ __forceinline__ FwdSeg fseg_then(const FwdSeg &X, const FwdSeg &Y) {
    if (Y.cl) return Y;
    return FwdSeg{X.P * Y.P, fma4(X.P, Y.S, X.S), X.cl};
}

template <int L, int LB>
__global__ void __launch_bounds__(256, 3) k_win_scan(const float *__restrict__ g, const float *__restrict__ c,
                                                  const float *__restrict__ a, float *__restrict__ R, int64_t T,
                                                  int N, int nslices, int64_t nseq, int64_t nchunks, int64_t W,
                                                  ScanWs d, unsigned *status) {
    __shared__ unsigned s_ticket;
    __shared__ float4 sP[SC_WARPS][32], sS[SC_WARPS][32], sCP[32], sCS[32];
    __shared__ bool sCl[SC_WARPS];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) s_ticket = atomicAdd(d.ticket, 1u);
    __syncthreads();
    const int64_t tk = s_ticket, chunk = tk / nseq, seq = tk % nseq;
    const int64_t b = seq / nslices;
    const int ch = int(seq % nslices) * SC_SLICE + lane * 4;
    const bool act = ch < N;
    const int64_t t0 = chunk * (SC_WARPS * L) + w * L;
    const int64_t base = b * T * N + ch;

    FwdSeg G{f4(1.f), f4(0.f), false};
    for (int k0 = 0; k0 < L; k0 += LB) {
        float4 av[LB], ev[LB];
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            const int64_t t = t0 + k0 + k;
            const bool ok = act && t < T;
            av[k] = ok ? ld_l2keep4(a + base + t * N) : f4(1.f);
            ev[k] = ok ? ld_l2keep4(g + base + t * N) * ld_l2keep4(c + base + t * N) : f4(0.f);
        }
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            const int64_t t = t0 + k0 + k;
            if (t >= T) break;
            if (t % W == 0) G = FwdSeg{f4(1.f), ev[k], true};
            else G = FwdSeg{G.P * av[k], fma4(G.P * av[k], ev[k], G.S), G.cl};
        }
    }
    sP[w][lane] = G.P;
    sS[w][lane] = G.S;
    if (lane == 0) sCl[w] = G.cl;
    __syncthreads();

    if (w == 0) {
        FwdSeg agg{sP[0][lane], sS[0][lane], sCl[0]};
#pragma unroll
        for (int j = 1; j < SC_WARPS; ++j) agg = fseg_then(agg, FwdSeg{sP[j][lane], sS[j][lane], sCl[j]});
        const int64_t di = seq * nchunks + chunk;
        // A closed aggregate is already the inclusive composite: publish it before looking
        // back.  The look-back still runs, for the tokens before the chunk's first block start.
        if (agg.cl) warp_publish(&d.inc0[di * 32 + lane], agg.P, &d.inc1[di * 32 + lane], agg.S, &d.flags[di], F_INC, lane);
        else warp_publish(&d.agg0[di * 32 + lane], agg.P, &d.agg1[di * 32 + lane], agg.S, &d.flags[di], F_AGG, lane);
        FwdSeg carry{f4(1.f), f4(0.f), true};
        if (chunk > 0) {
            const int64_t fb = seq * nchunks;
            carry = warp_lookback<FwdSeg>(
                d.flags + fb, chunk - 1, -1, chunk, FwdSeg{f4(1.f), f4(0.f), false},
                [&](int64_t p) { return FwdSeg{ld_cg4(&d.agg0[(fb + p) * 32 + lane]), ld_cg4(&d.agg1[(fb + p) * 32 + lane]), false}; },
                [&](int64_t p) { return FwdSeg{ld_cg4(&d.inc0[(fb + p) * 32 + lane]), ld_cg4(&d.inc1[(fb + p) * 32 + lane]), true}; },
                [](const FwdSeg &acc, const FwdSeg &g) { return fseg_then(g, acc); },
                [](const FwdSeg &acc, const FwdSeg &inc) { return fseg_then(inc, acc); },
                FwdSeg{f4(1.f), f4(0.f), true}, status, lane);
        }
        if (!agg.cl) {
            const FwdSeg inc = fseg_then(carry, agg);
            warp_publish(&d.inc0[di * 32 + lane], inc.P, &d.inc1[di * 32 + lane], inc.S, &d.flags[di], F_INC, lane);
        }
        sCP[lane] = carry.P;
        sCS[lane] = carry.S;
    }
    __syncthreads();

    G = FwdSeg{sCP[lane], sCS[lane], true};
    for (int j = 0; j < w; ++j) G = fseg_then(G, FwdSeg{sP[j][lane], sS[j][lane], sCl[j]});
    for (int k0 = 0; k0 < L; k0 += LB) {
        float4 av[LB], ev[LB];
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            const int64_t t = t0 + k0 + k;
            const bool ok = act && t < T;
            av[k] = ok ? ld_stream4(a + base + t * N) : f4(1.f);
            ev[k] = ok ? ld_stream4(g + base + t * N) * ld_stream4(c + base + t * N) : f4(0.f);
        }
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            const int64_t t = t0 + k0 + k;
            if (t >= T) break;
            if (t % W == 0) G = FwdSeg{f4(1.f), ev[k], true};
            else G = FwdSeg{G.P * av[k], fma4(G.P * av[k], ev[k], G.S), G.cl};
            if (act) st_stream4(R + base + t * N, G.S);
        }
    }
}

// ============================================================================ reverse adjoint scan
// Token i maps x (= mu_{i+1}) to b_i x + e_i with b_i = a_{i+1} (0 for the last token)
// and e_i = g_i c_i.  The composite of tokens i..j is x -> Q x + S.  A block-end token
// (i+1 multiple of W, or i = T-1) closes the composite: tokens after it do not reach i.
// Y after X (X earlier tokens) = X.closed ? X : (X.Q Y.Q, X.Q Y.S + X.S, Y.closed).
struct RevSeg {
    float4 Q, S;
    bool cl;
};
__device__ __forceinline__ RevSeg rseg_then(const RevSeg &X, const RevSeg &Y) {
    if (X.cl) return X;
    return RevSeg{X.Q * Y.Q, fma4(X.Q, Y.S, X.S), Y.cl};
}

template <int L, int LB, bool TRUNC, typename TD>
__global__ void __launch_bounds__(256, 3) k_bwd_scan(const float *__restrict__ g, const float *__restrict__ c,
                                                  const float *__restrict__ a, const float *__restrict__ h,
                                                  const float *__restrict__ R, TD *__restrict__ Da,
                                                  TD *__restrict__ Du, TD *__restrict__ Dc, TD *__restrict__ E,
                                                  int64_t T, int N, int nslices, int64_t nseq, int64_t nchunks,
                                                  int64_t W, ScanWs d, unsigned *status) {
    __shared__ unsigned s_ticket;
    __shared__ float4 sQ[SC_WARPS][32], sS[SC_WARPS][32], sCQ[32], sCS[32];
    __shared__ bool sCl[SC_WARPS];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) s_ticket = atomicAdd(d.ticket, 1u);
    __syncthreads();
    const int64_t tk = s_ticket, chunk = nchunks - 1 - tk / nseq, seq = tk % nseq;
    const int64_t b = seq / nslices;
    const int ch = int(seq % nslices) * SC_SLICE + lane * 4;
    const bool act = ch < N;
    const int64_t t0 = chunk * (SC_WARPS * L) + w * L;
    const int64_t base = b * T * N + ch;

    // pass 1: composite of this thread's tokens from e_i = g_i c_i and b_i = a_{i+1}
    // (0 past the last token); the rows stay in L2 for pass 2.
    RevSeg G{f4(1.f), f4(0.f), false};
    for (int k0 = L - LB; k0 >= 0; k0 -= LB) {
        float4 ev[LB], bv[LB];
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            const int64_t t = t0 + k0 + k;
            const bool ok = act && t < T;
            ev[k] = ok ? ld_l2keep4(g + base + t * N) * ld_l2keep4(c + base + t * N) : f4(0.f);
            bv[k] = (act && t + 1 < T) ? ld_l2keep4(a + base + (t + 1) * N) : f4(0.f);
        }
#pragma unroll
        for (int k = LB - 1; k >= 0; --k) {
            const int64_t t = t0 + k0 + k;
            if (t >= T) continue;
            const bool end = (t == T - 1) || (TRUNC && (t + 1) % W == 0);
            if (end) G = RevSeg{bv[k], ev[k], true};
            else G = RevSeg{bv[k] * G.Q, fma4(bv[k], G.S, ev[k]), G.cl};
        }
    }
    sQ[w][lane] = G.Q;
    sS[w][lane] = G.S;
    if (lane == 0) sCl[w] = G.cl;
    __syncthreads();

    if (w == 0) {
        RevSeg agg{sQ[0][lane], sS[0][lane], sCl[0]};
#pragma unroll
        for (int j = 1; j < SC_WARPS; ++j) agg = rseg_then(agg, RevSeg{sQ[j][lane], sS[j][lane], sCl[j]});
        const int64_t di = seq * nchunks + chunk;
        // A closed aggregate is already the inclusive composite: publish it before looking
        // back.  The look-back still runs, for the tokens after the chunk's last block end.
        if (agg.cl) warp_publish(&d.inc0[di * 32 + lane], agg.Q, &d.inc1[di * 32 + lane], agg.S, &d.flags[di], F_INC, lane);
        else warp_publish(&d.agg0[di * 32 + lane], agg.Q, &d.agg1[di * 32 + lane], agg.S, &d.flags[di], F_AGG, lane);
        RevSeg carry{f4(0.f), f4(0.f), true};
        if (chunk + 1 < nchunks) {
            const int64_t fb = seq * nchunks;
            carry = warp_lookback<RevSeg>(
                d.flags + fb, chunk + 1, 1, nchunks - 1 - chunk, RevSeg{f4(1.f), f4(0.f), false},
                [&](int64_t p) { return RevSeg{ld_cg4(&d.agg0[(fb + p) * 32 + lane]), ld_cg4(&d.agg1[(fb + p) * 32 + lane]), false}; },
                [&](int64_t p) { return RevSeg{ld_cg4(&d.inc0[(fb + p) * 32 + lane]), ld_cg4(&d.inc1[(fb + p) * 32 + lane]), true}; },
                [](const RevSeg &acc, const RevSeg &g) { return rseg_then(acc, g); },
                [](const RevSeg &acc, const RevSeg &inc) { return rseg_then(acc, inc); },
                RevSeg{f4(0.f), f4(0.f), true}, status, lane);
        }
        if (!agg.cl) {
            const RevSeg inc = rseg_then(agg, carry);
            warp_publish(&d.inc0[di * 32 + lane], inc.Q, &d.inc1[di * 32 + lane], inc.S, &d.flags[di], F_INC, lane);
        }
        sCQ[lane] = carry.Q;
        sCS[lane] = carry.S;
    }
    __syncthreads();

    // composite of everything after this warp's tokens, then pass 2 backwards
    G = RevSeg{sCQ[lane], sCS[lane], true};
    for (int j = SC_WARPS - 1; j > w; --j) G = rseg_then(RevSeg{sQ[j][lane], sS[j][lane], sCl[j]}, G);
    // rows: a at t0..t0+L, h at t0-1..t0+L-1, g and c at t0..t0+L-1
    float4 anext = (act && t0 + L < T) ? ld_keep4(a + base + (t0 + L) * N) : f4(0.f);
#pragma unroll
    for (int k = L - 1; k >= 0; --k) {
        const int64_t t = t0 + k;
        if (t >= T) continue;
        const float4 gk = act ? ld_stream4(g + base + t * N) : f4(0.f);
        const float4 ck = act ? ld_stream4(c + base + t * N) : f4(0.f);
        const float4 ak = act ? ld_keep4(a + base + t * N) : f4(0.f);
        const float4 hk = act ? ld_keep4(h + base + t * N) : f4(0.f);
        const float4 hp = (act && t > 0) ? ld_keep4(h + base + (t - 1) * N) : f4(0.f);
        const float4 bk = t + 1 < T ? anext : f4(0.f);
        const float4 ek = gk * ck;
        const bool end = (t == T - 1) || (TRUNC && (t + 1) % W == 0);
        if (end) G = RevSeg{bk, ek, true};
        else G = RevSeg{bk * G.Q, fma4(bk, G.S, ek), true};
        float4 mu = G.S;
        if (TRUNC && act && t % W != 0 && (t / W + 1) * W < T) {
            const int64_t m = t + W - 1 < T - 1 ? t + W - 1 : T - 1;
            mu = fma4(G.Q, ld_stream4(R + base + m * N), G.S);
        }
        if (act) {
            st4(Dc + base + t * N, gk * hk);
            st4(E + base + t * N, ck * hk);
            st4(Du + base + t * N, mu);
            st4(Da + base + t * N, mu * hp * ak * (f4(1.f) - ak));
        }
        anext = ak;
    }
}

// ============================================================================ launchers
cudaError_t launch_fwd_scan(const float *a, const float *u, float *h, int64_t B, int64_t T, int N,
                            void *scan_ws, unsigned *status, cudaStream_t st) {
    constexpr int L = 16, LB = 8;
    const int nslices = int(cdiv(N, SC_SLICE));
    const int64_t nseq = B * nslices, nchunks = cdiv(T, SC_WARPS * L);
    ScanWs d = scan_ws_carve(scan_ws, B, T, N);
    cudaError_t e = cudaMemsetAsync(scan_ws, 0, scan_reset_bytes(B, T, N), st);
    if (e != cudaSuccess) return e;
    k_fwd_scan<L, LB><<<unsigned(nseq * nchunks), 256, 0, st>>>(a, u, h, T, N, nslices, nseq, nchunks, d, status);
    return cudaGetLastError();
}

cudaError_t launch_win_scan(const float *g, const float *c, const float *a, float *R, int64_t B,
                            int64_t T, int N, int64_t W, void *scan_ws, unsigned *status, cudaStream_t st) {
    constexpr int L = 16, LB = 4;
    const int nslices = int(cdiv(N, SC_SLICE));
    const int64_t nseq = B * nslices, nchunks = cdiv(T, SC_WARPS * L);
    ScanWs d = scan_ws_carve(scan_ws, B, T, N);
    cudaError_t e = cudaMemsetAsync(scan_ws, 0, scan_reset_bytes(B, T, N), st);
    if (e != cudaSuccess) return e;
    k_win_scan<L, LB><<<unsigned(nseq * nchunks), 256, 0, st>>>(g, c, a, R, T, N, nslices, nseq, nchunks, W, d, status);
    return cudaGetLastError();
}

cudaError_t launch_bwd_scan(const float *g, const float *c, const float *a, const float *h, const float *R,
                            void *D_a, void *D_u, void *D_c, void *E, bool d_bf16, int64_t B, int64_t T, int N,
                            int64_t W, void *scan_ws, unsigned *status, cudaStream_t st) {
    constexpr int L = 16, LB = 4;
    const int nslices = int(cdiv(N, SC_SLICE));
    const int64_t nseq = B * nslices, nchunks = cdiv(T, SC_WARPS * L);
    ScanWs d = scan_ws_carve(scan_ws, B, T, N);
    cudaError_t e = cudaMemsetAsync(scan_ws, 0, scan_reset_bytes(B, T, N), st);
    if (e != cudaSuccess) return e;
    const bool trunc = W > 0 && W < T;
    const unsigned grid = unsigned(nseq * nchunks);
#define ADJ_BWD(TR, TD)                                                                                      \
    k_bwd_scan<L, LB, TR, TD><<<grid, 256, 0, st>>>(g, c, a, h, R, static_cast<TD *>(D_a), static_cast<TD *>(D_u), \
                                                static_cast<TD *>(D_c), static_cast<TD *>(E), T, N, nslices,   \
                                                nseq, nchunks, trunc ? W : T, d, status)
    if (d_bf16) {
        if (trunc) ADJ_BWD(true, __nv_bfloat16);
        else ADJ_BWD(false, __nv_bfloat16);
    } else {
        if (trunc) ADJ_BWD(true, float);
        else ADJ_BWD(false, float);
    }
#undef ADJ_BWD
    return cudaGetLastError();
}

}  // namespace adj
