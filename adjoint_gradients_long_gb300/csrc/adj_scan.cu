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
// Work decomposition (all three kernels): a CTA of 8 warps owns one chunk of 8*L
// consecutive tokens of one sequence and 128 channels.  The chunk's input rows are
// staged in shared memory by one TMA load per array (rows of 128 fp32, 512 bytes), so
// both passes read them from shared memory and HBM sees every input byte once.  Lane
// = 4 channels (one float4 per token row), warp w = tokens [w*L, (w+1)*L) of the
// chunk.  Pass 1 reduces each thread's L tokens to one composite map; the 8 warp
// composites are combined in shared memory and warp 0 publishes the chunk aggregate;
// the CTA then looks back over its predecessors' descriptors (decoupled look-back).
// Pass 2 applies the carry and writes the outputs.  Chunks are numbered by an atomic
// ticket in scan order, so a CTA only ever waits for CTAs that started before it; every
// wait is bounded.
//
// Descriptors carry no flags: before each launch every descriptor word is set to the
// bit pattern 0xFFFFFFFF, a NaN that no arithmetic produces (results that are NaN come
// out as the canonical 0x7FFFFFFF, and published values are canonicalised), and each
// word is written exactly once per launch.  A reader that sees no sentinel in a
// descriptor therefore holds its published value, so one L2 round trip both finds and
// reads a predecessor's aggregate or inclusive prefix, and publishing needs no fence.
#include <string.h>

#include "adj_internal.cuh"
#include "adj_ptx.cuh"
#include "adj_tmap.cuh"

namespace adj {

constexpr int SC_WARPS = 8;
#ifndef ADJ_SCAN_FWD_L
#define ADJ_SCAN_FWD_L 12
#endif
#ifndef ADJ_SCAN_BWD_L
#define ADJ_SCAN_BWD_L 8
#endif
#ifndef ADJ_SCAN_TRUNC_L
#define ADJ_SCAN_TRUNC_L 8
#endif
// tokens per warp (chunk = 8 L tokens) of the forward scan, of the window and reverse scans,
// and of the one-pass truncated adjoint
constexpr int SC_FWD_L = ADJ_SCAN_FWD_L, SC_BWD_L = ADJ_SCAN_BWD_L, SC_TRUNC_L = ADJ_SCAN_TRUNC_L;
constexpr int SC_SLICE = 128;        // channels per CTA
constexpr int SC_MIN_CHUNK = 32;     // smallest chunk (L = 4); sizes the descriptor arrays
constexpr unsigned SC_EMPTY = 0xFFFFFFFFu;   // descriptor word not yet published

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t scan_ws_bytes(int64_t B, int64_t T, int N) {
    int64_t n = B * cdiv(N, SC_SLICE) * cdiv(T, SC_MIN_CHUNK);
    return 256 + 4 * size_t(n) * 32 * sizeof(float4);
}

// Ticket, then the four descriptor arrays of n = nseq * nchunks chunks, back to back.
ScanWs scan_ws_carve(void *base, int64_t n) {
    char *p = static_cast<char *>(base);
    ScanWs d;
    d.ticket = reinterpret_cast<unsigned *>(p);
    p += 256;
    const size_t db = size_t(n) * 32 * sizeof(float4);
    d.agg0 = reinterpret_cast<float4 *>(p); p += db;
    d.agg1 = reinterpret_cast<float4 *>(p); p += db;
    d.inc0 = reinterpret_cast<float4 *>(p); p += db;
    d.inc1 = reinterpret_cast<float4 *>(p);
    return d;
}

// Before a launch over n chunks, one memset: every descriptor word empty, and the ticket
// 0xFFFFFFFF (a CTA's chunk is the value it read plus one).
static cudaError_t scan_ws_reset(void *base, int64_t n, cudaStream_t st) {
    return cudaMemsetAsync(base, 0xFF, 256 + 4 * size_t(n) * 32 * sizeof(float4), st);
}

__device__ __forceinline__ float canon(float x) {
    return __float_as_uint(x) == SC_EMPTY ? __uint_as_float(0x7FFFFFFFu) : x;
}
__device__ __forceinline__ float4 canon4(float4 v) { return make_float4(canon(v.x), canon(v.y), canon(v.z), canon(v.w)); }
__device__ __forceinline__ bool full4(float4 v) {
    return __float_as_uint(v.x) != SC_EMPTY && __float_as_uint(v.y) != SC_EMPTY && __float_as_uint(v.z) != SC_EMPTY &&
           __float_as_uint(v.w) != SC_EMPTY;
}
// Publish one or two float4 per lane (p1 may be null); no fence, no flag.
__device__ __forceinline__ void desc_publish(float4 *p0, float4 v0, float4 *p1, float4 v1) {
    if (p0) st_cg4(p0, canon4(v0));
    if (p1) st_cg4(p1, canon4(v1));
}
// A descriptor slot as read: the value and whether every word of it was published.
struct DescRead {
    float4 a, b;
    bool ok;
};
__device__ __forceinline__ DescRead desc_read(const float4 *p0, const float4 *p1) {
    DescRead r;
    r.a = p0 ? ld_cg4(p0) : f4(0.f);
    r.b = ld_cg4(p1);
    r.ok = (!p0 || full4(r.a)) && full4(r.b);
    return r;
}

// ============================================================================ segment composites
// Composite maps of token ranges (see each scan below).  Each packs into two float4
// and a closed flag, so a CTA can pass them through shared memory.
struct float2x4 {   // forward state scan: h_out = x h_in + y
    float4 x, y;
};
struct FwdSeg {     // window scan R
    float4 P, S;
    bool cl;
};
struct RevSeg {     // reverse adjoint scan
    float4 Q, S;
    bool cl;
};
__device__ __forceinline__ void seg_put(const float2x4 &c, float4 &a, float4 &b, bool &cl) { a = c.x; b = c.y; cl = false; }
__device__ __forceinline__ void seg_put(const FwdSeg &c, float4 &a, float4 &b, bool &cl) { a = c.P; b = c.S; cl = c.cl; }
__device__ __forceinline__ void seg_put(const RevSeg &c, float4 &a, float4 &b, bool &cl) { a = c.Q; b = c.S; cl = c.cl; }
__device__ __forceinline__ void seg_get(float2x4 &c, float4 a, float4 b, bool) { c = float2x4{a, b}; }
__device__ __forceinline__ void seg_get(FwdSeg &c, float4 a, float4 b, bool cl) { c = FwdSeg{a, b, cl}; }
__device__ __forceinline__ void seg_get(RevSeg &c, float4 a, float4 b, bool cl) { c = RevSeg{a, b, cl}; }

// CTA-wide decoupled look-back (all threads call it).  Each round, warp j reads the
// descriptors (aggregate and inclusive prefix) of predecessors done + 2j and
// done + 2j + 1 (nearest first: p0, p0 + dir, ...), all sixteen in flight at once, and
// folds them in order until an inclusive prefix (closed: the fold ends there), a
// predecessor that has published nothing yet, or the end of the sequence (folds
// zero_inc).  Warp 0 then folds the warps' partial composites in warp order up to the
// first warp that stopped; a round costs one L2 round trip.  extend(acc, x) composes one
// more (older) predecessor, or an inclusive prefix, into acc.  load(p) returns the slot's
// aggregate and inclusive prefix as read.  sx, sy, scl (8 x 32) and ctl (8 + 2 words) are
// shared scratch.  The carry is valid in warp 0; a wait that gives up records the timeout
// and finishes with zero_inc (so does one that sees another CTA's recorded timeout).
constexpr int LB_PER = 2;   // predecessors a warp examines per round
template <class C, class LD, class EX>
__device__ __forceinline__ C cta_lookback(int64_t p0, int dir, int64_t count, C ident, LD load, EX extend, C zero_inc,
                                          unsigned *status, float4 (*sx)[32], float4 (*sy)[32], bool *scl, int *ctl,
                                          int w, int lane) {
    C acc = ident;
    int64_t done = 0;
    for (int round = 0; round < SPIN_LIMIT; ++round) {
        // this warp's predecessors: all loads first
        C ag[LB_PER], ic[LB_PER];
        bool aok[LB_PER], iok[LB_PER];
#pragma unroll
        for (int i = 0; i < LB_PER; ++i) {
            const int64_t j = done + LB_PER * w + i;
            aok[i] = iok[i] = false;
            if (j < count) load(p0 + dir * j, ag[i], aok[i], ic[i], iok[i]);
        }
        C part = ident;
        int stop = 0;   // 0: all folded, 1: closed (inclusive prefix or sequence end), 2: missing
        int used = 0;
#pragma unroll
        for (int i = 0; i < LB_PER; ++i) {
            if (stop) break;
            const int64_t j = done + LB_PER * w + i;
            if (j >= count) {
                part = extend(part, zero_inc);
                stop = 1;
            } else if (__all_sync(0xffffffffu, iok[i])) {
                part = extend(part, ic[i]);
                stop = 1;
            } else if (__all_sync(0xffffffffu, aok[i])) {
                part = extend(part, ag[i]);
                ++used;
            } else {
                stop = 2;
            }
        }
        bool cl;
        seg_put(part, sx[w][lane], sy[w][lane], cl);
        if (lane == 0) {
            scl[w] = cl;
            ctl[w] = stop | (used << 4);
        }
        __syncthreads();
        if (w == 0) {
            int state = 0;   // 0: more rounds, 1: done, 2: poll again
            int64_t adv = 0;
            for (int j = 0; j < SC_WARPS; ++j) {
                const int st = ctl[j] & 15, u = ctl[j] >> 4;
                C pj;
                seg_get(pj, sx[j][lane], sy[j][lane], scl[j]);
                acc = extend(acc, pj);
                adv += u;
                if (st == 1) {
                    state = 1;
                    break;
                }
                if (st == 2) {
                    state = 2;
                    break;
                }
            }
            // still waiting: give up early once any CTA has recorded a timeout (the
            // predecessor may never publish)
            if (state == 2 && (round & 255) == 255 && *reinterpret_cast<volatile unsigned *>(status) != 0u)
                state = 3;
            if (lane == 0) {
                ctl[SC_WARPS] = state;
                ctl[SC_WARPS + 1] = int(adv);
            }
        }
        __syncthreads();
        const int state = ctl[SC_WARPS];
        done += ctl[SC_WARPS + 1];
        if (state == 1) return acc;
        if (state == 3) return extend(acc, zero_inc);
        if (state == 2 && round > 8) __nanosleep(64);
    }
    record_timeout(status);
    return extend(acc, zero_inc);
}

// ============================================================================ chunk staging
// Up to four input arrays of a scan, each a TMA map over [B*T rows, N cols] fp32 with a
// box of 128 channels x (rows of the chunk).
struct ScanMaps {
    CUtensorMap m[4];
};

__device__ __forceinline__ float *smem_1k(uint8_t *p) {
    return reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Take the chunk ticket and set up the staging barrier (thread 0), then the CTA syncs.
__device__ __forceinline__ unsigned chunk_ticket(const ScanWs &d, unsigned *s_ticket, uint64_t *bar, int *abort_flag) {
    if (threadIdx.x == 0) {
        *s_ticket = atomicAdd(d.ticket, 1u) + 1u;   // the reset leaves 0xFFFFFFFF: first ticket 0
        mbar_init(smem_u32(bar), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    return *s_ticket;
}

// Thread 0: load rows [y, y + rows_i) x channels [x, x + 128) of map i into dst_i
// (n arrays), all counted on one barrier.  Rows past the array read as zero.
__device__ __forceinline__ void stage_chunk(const ScanMaps &mp, int n, float *const *dst, const int *rows, int x,
                                            int64_t y, uint64_t *bar) {
    if (threadIdx.x != 0) return;
    uint32_t bytes = 0;
    for (int i = 0; i < n; ++i) bytes += uint32_t(rows[i]) * SC_SLICE * 4u;
    mbar_arrive_expect_tx(smem_u32(bar), bytes);
    for (int i = 0; i < n; ++i) tma_load_2d(smem_u32(dst[i]), &mp.m[i], x, int(y), smem_u32(bar));
}

// Row r of a staged array as this lane's float4.
__device__ __forceinline__ float4 srow(const float *s, int r, int lane) {
    return *reinterpret_cast<const float4 *>(s + r * SC_SLICE + lane * 4);
}

// ============================================================================ forward state scan
// Composite of a token range: h_out = A h_in + H.  (A2,H2) after (A1,H1) = (A2 A1, A2 H1 + H2).
// Staged: a and u, rows [c0, c0 + 8L).  With EOUT the scan also writes chx = c . h rounded
// to bf16 (the output projection's operand in bf16 layers), reading c from global memory
// (its loads issued before the staging wait).
template <int L, bool EOUT>
__global__ void __launch_bounds__(256, (L <= 6 ? 4 : L <= 8 ? 3 : L <= 12 ? 2 : 1)) k_fwd_scan(const __grid_constant__ ScanMaps mp, float *__restrict__ h,
                                                  const float *__restrict__ c, __nv_bfloat16 *__restrict__ chx,
                                                  int64_t T, int N, int nslices, int64_t nseq, int64_t nchunks,
                                                  ScanWs d, unsigned *status) {
    constexpr int TT = SC_WARPS * L;
    extern __shared__ uint8_t sm_dyn[];
    float *sa = smem_1k(sm_dyn), *su = sa + TT * SC_SLICE;
    __shared__ unsigned s_ticket;
    __shared__ uint64_t s_bar;
    __shared__ int s_abort;
    __shared__ float4 sA[SC_WARPS][32], sH[SC_WARPS][32], sC[32];
    __shared__ bool s_cl[SC_WARPS];
    __shared__ int s_ctl[SC_WARPS + 2];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tk = chunk_ticket(d, &s_ticket, &s_bar, &s_abort), chunk = tk / nseq, seq = tk % nseq;
    const int64_t b = seq / nslices;
    const int slice = int(seq % nslices), ch = slice * SC_SLICE + lane * 4;
    const bool act = ch < N;
    const int64_t c0 = chunk * TT, t0 = c0 + w * L;
    {
        float *dst[2] = {sa, su};
        const int rows[2] = {TT, TT};
        stage_chunk(mp, 2, dst, rows, slice * SC_SLICE, b * T + c0, &s_bar);
    }
    const int64_t base = b * T * N + ch;
    float4 cv[EOUT ? L : 1];
    if (EOUT) {
#pragma unroll
        for (int k = 0; k < L; ++k) cv[k] = (act && t0 + k < T) ? ld_stream4(c + base + (t0 + k) * N) : f4(0.f);
    }
    mbar_wait(smem_u32(&s_bar), 0, &s_abort, status);

    // pass 1: composite of this thread's L tokens
    float4 A = f4(1.f), H = f4(0.f);
#pragma unroll
    for (int k = 0; k < L; ++k) {
        if (t0 + k >= T) break;
        const float4 av = srow(sa, w * L + k, lane), uv = srow(su, w * L + k, lane);
        H = fma4(av, H, uv);
        A = A * av;
    }
    sA[w][lane] = A;
    sH[w][lane] = H;
    __syncthreads();

    // this warp's prefix (warps before it) and, in warp 0, the chunk aggregate
    float4 pA = f4(1.f), pH = f4(0.f);
    for (int j = 0; j < w; ++j) {
        pH = fma4(sA[j][lane], pH, sH[j][lane]);
        pA = pA * sA[j][lane];
    }
    float4 cA = f4(1.f), cH = f4(0.f);
    const int64_t di = seq * nchunks + chunk, fb = seq * nchunks;
    if (w == 0) {
#pragma unroll
        for (int j = 0; j < SC_WARPS; ++j) {
            cH = fma4(sA[j][lane], cH, sH[j][lane]);
            cA = cA * sA[j][lane];
        }
        if (chunk > 0) desc_publish(&d.agg0[di * 32 + lane], cA, &d.agg1[di * 32 + lane], cH);
    }
    __syncthreads();   // sA/sH now serve as look-back scratch
    float4 carry = f4(0.f);
    if (chunk > 0) {
        // acc = composite of the chunks between the inclusive prefix found and this chunk
        const float2x4 r = cta_lookback<float2x4>(
            chunk - 1, -1, chunk, float2x4{f4(1.f), f4(0.f)},
            [&](int64_t p, float2x4 &ag, bool &aok, float2x4 &ic, bool &iok) {
                const DescRead A = desc_read(&d.agg0[(fb + p) * 32 + lane], &d.agg1[(fb + p) * 32 + lane]);
                const DescRead I = desc_read(nullptr, &d.inc1[(fb + p) * 32 + lane]);
                ag = float2x4{A.a, A.b};
                aok = A.ok;
                ic = float2x4{f4(0.f), I.b};   // inclusive: h at the chunk end, closed
                iok = I.ok;
            },
            [](const float2x4 &acc, const float2x4 &g) { return float2x4{acc.x * g.x, fma4(acc.x, g.y, acc.y)}; },
            float2x4{f4(0.f), f4(0.f)}, status, sA, sH, s_cl, s_ctl, w, lane);
        carry = r.y;
    }
    if (w == 0) {
        desc_publish(nullptr, f4(0.f), &d.inc1[di * 32 + lane], fma4(cA, carry, cH));
        sC[lane] = carry;
    }
    __syncthreads();

    // pass 2: h from the carry into this warp's first token
    float4 hc = fma4(pA, sC[lane], pH);
#pragma unroll
    for (int k = 0; k < L; ++k) {
        const int64_t t = t0 + k;
        if (t >= T) break;
        hc = fma4(srow(sa, w * L + k, lane), hc, srow(su, w * L + k, lane));
        if (act) {
            st4(h + base + t * N, hc);   // kept in L2 (the output projection reads c . h next)
            if (EOUT) st4(chx + base + t * N, cv[k] * hc);
        }
    }
}

// ============================================================================ window scan R
// Forward scan restarted at every multiple of W.  Token m maps the state (P, R) to
// (a_m P, R + e_m a_m P); a block-start token resets it to (1, e_m).  Composite of a
// range: (Pi, Sig, closed); Y after X = Y.closed ? Y : (X.Pi Y.Pi, X.Sig + X.Pi Y.Sig, X.closed).
// Output R_m = Sig of the composite from the block start to m.
__device__ __forceinline__ FwdSeg fseg_then(const FwdSeg &X, const FwdSeg &Y) {
    if (Y.cl) return Y;
    return FwdSeg{X.P * Y.P, fma4(X.P, Y.S, X.S), X.cl};
}

// Staged: g, c and a, rows [c0, c0 + 8L).
template <int L>
__global__ void __launch_bounds__(256, (L <= 4 ? 4 : L <= 6 ? 3 : L <= 8 ? 2 : 1)) k_win_scan(const __grid_constant__ ScanMaps mp, float *__restrict__ R,
                                                  int64_t T, int N, int nslices, int64_t nseq, int64_t nchunks,
                                                  int64_t W, ScanWs d, unsigned *status) {
    constexpr int TT = SC_WARPS * L;
    extern __shared__ uint8_t sm_dyn[];
    float *sg = smem_1k(sm_dyn), *sc = sg + TT * SC_SLICE, *sa = sc + TT * SC_SLICE;
    __shared__ unsigned s_ticket;
    __shared__ uint64_t s_bar;
    __shared__ int s_abort;
    __shared__ float4 sP[SC_WARPS][32], sS[SC_WARPS][32], sCP[32], sCS[32];
    __shared__ bool sCl[SC_WARPS];
    __shared__ int s_ctl[SC_WARPS + 2];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tk = chunk_ticket(d, &s_ticket, &s_bar, &s_abort), chunk = tk / nseq, seq = tk % nseq;
    const int64_t b = seq / nslices;
    const int slice = int(seq % nslices), ch = slice * SC_SLICE + lane * 4;
    const bool act = ch < N;
    const int64_t c0 = chunk * TT, t0 = c0 + w * L;
    {
        float *dst[3] = {sg, sc, sa};
        const int rows[3] = {TT, TT, TT};
        stage_chunk(mp, 3, dst, rows, slice * SC_SLICE, b * T + c0, &s_bar);
    }
    mbar_wait(smem_u32(&s_bar), 0, &s_abort, status);

    FwdSeg G{f4(1.f), f4(0.f), false};
#pragma unroll
    for (int k = 0; k < L; ++k) {
        const int64_t t = t0 + k;
        if (t >= T) break;
        const int r = w * L + k;
        const float4 ev = srow(sg, r, lane) * srow(sc, r, lane), av = srow(sa, r, lane);
        if (t % W == 0) G = FwdSeg{f4(1.f), ev, true};
        else G = FwdSeg{G.P * av, fma4(G.P * av, ev, G.S), G.cl};
    }
    sP[w][lane] = G.P;
    sS[w][lane] = G.S;
    if (lane == 0) sCl[w] = G.cl;
    __syncthreads();

    // this warp's prefix (warps before it) and, in warp 0, the chunk aggregate
    FwdSeg pre{f4(1.f), f4(0.f), false};
    for (int j = 0; j < w; ++j) pre = fseg_then(pre, FwdSeg{sP[j][lane], sS[j][lane], sCl[j]});
    FwdSeg agg{sP[0][lane], sS[0][lane], sCl[0]};
    const int64_t di = seq * nchunks + chunk, fb = seq * nchunks;
    if (w == 0) {
#pragma unroll
        for (int j = 1; j < SC_WARPS; ++j) agg = fseg_then(agg, FwdSeg{sP[j][lane], sS[j][lane], sCl[j]});
        // A closed aggregate is already the inclusive composite: publish it before looking
        // back.  The look-back still runs, for the tokens before the chunk's first block start.
        if (agg.cl) desc_publish(&d.inc0[di * 32 + lane], agg.P, &d.inc1[di * 32 + lane], agg.S);
        else desc_publish(&d.agg0[di * 32 + lane], agg.P, &d.agg1[di * 32 + lane], agg.S);
    }
    __syncthreads();   // sP/sS/sCl now serve as look-back scratch
    FwdSeg carry{f4(1.f), f4(0.f), true};
    if (chunk > 0) {
        carry = cta_lookback<FwdSeg>(
            chunk - 1, -1, chunk, FwdSeg{f4(1.f), f4(0.f), false},
            [&](int64_t p, FwdSeg &ag, bool &aok, FwdSeg &ic, bool &iok) {
                const DescRead A = desc_read(&d.agg0[(fb + p) * 32 + lane], &d.agg1[(fb + p) * 32 + lane]);
                const DescRead I = desc_read(&d.inc0[(fb + p) * 32 + lane], &d.inc1[(fb + p) * 32 + lane]);
                ag = FwdSeg{A.a, A.b, false};
                aok = A.ok;
                ic = FwdSeg{I.a, I.b, true};
                iok = I.ok;
            },
            [](const FwdSeg &acc, const FwdSeg &g) { return fseg_then(g, acc); },
            FwdSeg{f4(1.f), f4(0.f), true}, status, sP, sS, sCl, s_ctl, w, lane);
    }
    if (w == 0) {
        if (!agg.cl) {
            const FwdSeg inc = fseg_then(carry, agg);
            desc_publish(&d.inc0[di * 32 + lane], inc.P, &d.inc1[di * 32 + lane], inc.S);
        }
        sCP[lane] = carry.P;
        sCS[lane] = carry.S;
    }
    __syncthreads();

    G = fseg_then(FwdSeg{sCP[lane], sCS[lane], true}, pre);
    const int64_t base = b * T * N + ch;
#pragma unroll
    for (int k = 0; k < L; ++k) {
        const int64_t t = t0 + k;
        if (t >= T) break;
        const int r = w * L + k;
        const float4 ev = srow(sg, r, lane) * srow(sc, r, lane), av = srow(sa, r, lane);
        if (t % W == 0) G = FwdSeg{f4(1.f), ev, true};
        else G = FwdSeg{G.P * av, fma4(G.P * av, ev, G.S), G.cl};
        if (act) st4(R + base + t * N, G.S);   // kept in L2: the reverse scan reads R next
    }
}

// ============================================================================ reverse adjoint scan
// Token i maps x (= mu_{i+1}) to b_i x + e_i with b_i = a_{i+1} (0 for the last token)
// and e_i = g_i c_i.  The composite of tokens i..j is x -> Q x + S.  A block-end token
// (i+1 multiple of W, or i = T-1) closes the composite: tokens after it do not reach i.
// Y after X (X earlier tokens) = X.closed ? X : (X.Q Y.Q, X.Q Y.S + X.S, Y.closed).
__device__ __forceinline__ RevSeg rseg_then(const RevSeg &X, const RevSeg &Y) {
    if (X.cl) return X;
    return RevSeg{X.Q * Y.Q, fma4(X.Q, Y.S, X.S), Y.cl};
}

// A seed as the parameter GEMMs read it (rounded to its storage type).
template <typename TD>
__device__ __forceinline__ float4 as_stored(float4 v) {
    if constexpr (sizeof(TD) == 2) {
        return make_float4(__bfloat162float(__float2bfloat16_rn(v.x)), __bfloat162float(__float2bfloat16_rn(v.y)),
                           __bfloat162float(__float2bfloat16_rn(v.z)), __bfloat162float(__float2bfloat16_rn(v.w)));
    } else {
        return v;
    }
}
__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }
// Sums of eight values over the 32 lanes of a warp in 9 shuffles: each exchange halves the
// values a lane keeps.  Returns, in every lane, the total of value
// k = 4 (lane >> 4 & 1) + 2 (lane >> 3 & 1) + (lane >> 2 & 1).
__device__ __forceinline__ float warp_sum8(const float (&v)[8], int lane) {
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = (h16 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, h16 ? v[i] : v[i + 4], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i) b[i] = (h8 ? a[i + 2] : a[i]) + __shfl_xor_sync(0xffffffffu, h8 ? a[i] : a[i + 2], 8);
    float c = (h4 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, h4 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
}
__device__ __forceinline__ int warp_sum8_index(int lane) { return 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1); }

// z = logit(a) - b (the gate's pre-activation xhat W_a); 0 where a is 0 or 1, where the
// gate seed a (1 - a) vanishes
__device__ __forceinline__ float gate_z(float a, float b) {
    return (a > 0.f && a < 1.f) ? __logf(__fdividef(a, 1.f - a)) - b : 0.f;
}

// Staged: g and c, rows [c0, c0 + 8L), and a, rows [c0, c0 + 8L] (one more: b of the
// chunk's last token).  h (and R) are read from global memory, their loads issued
// before the staging wait.  D_c and E are written right after pass 1, before the
// look-back; D_u and D_a in pass 2.
// DZ: also dz[token][slice] = sum over the slice's channels of D_a z_a + D_u u + D_c c
// (seeds as stored; z_a = logit(a) - b_a, u_t = h_t - a_t h_{t-1}): with z = xhat W_in
// this is D . (xhat W_in) = xhat . (D W_in^T) = xhat . dxhat, the row dot product that the
// cotangent through a normalised layer input needs, without reading dxhat.
template <int L, bool TRUNC, typename TD, bool DZ = false>
__global__ void __launch_bounds__(256, (L <= 4 ? 4 : L <= 6 ? 3 : L <= 8 ? 2 : 1)) k_bwd_scan(const __grid_constant__ ScanMaps mp, const float *__restrict__ h,
                                                  const float *__restrict__ R, TD *__restrict__ Da,
                                                  TD *__restrict__ Du, TD *__restrict__ Dc, TD *__restrict__ E,
                                                  int64_t T, int N, int nslices, int64_t nseq, int64_t nchunks,
                                                  int64_t W, ScanWs d, unsigned *status,
                                                  const float *__restrict__ b_a, float *__restrict__ dz) {
    constexpr int TT = SC_WARPS * L;
    extern __shared__ uint8_t sm_dyn[];
    float *sg = smem_1k(sm_dyn), *sc = sg + TT * SC_SLICE, *sa = sc + TT * SC_SLICE;
    __shared__ unsigned s_ticket;
    __shared__ uint64_t s_bar;
    __shared__ int s_abort;
    __shared__ float4 sQ[SC_WARPS][32], sS[SC_WARPS][32], sCQ[32], sCS[32];
    __shared__ bool sCl[SC_WARPS];
    __shared__ int s_ctl[SC_WARPS + 2];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tk = chunk_ticket(d, &s_ticket, &s_bar, &s_abort), chunk = nchunks - 1 - tk / nseq, seq = tk % nseq;
    const int64_t b = seq / nslices;
    const int slice = int(seq % nslices), ch = slice * SC_SLICE + lane * 4;
    const bool act = ch < N;
    const int64_t c0 = chunk * TT, t0 = c0 + w * L;
    const int64_t base = b * T * N + ch;
    {
        float *dst[3] = {sg, sc, sa};
        const int rows[3] = {TT, TT, TT + 1};
        stage_chunk(mp, 3, dst, rows, slice * SC_SLICE, b * T + c0, &s_bar);
    }
    // h_{t-1} and h_t of this thread's tokens, from global
    float4 hv[L + 1];
    hv[0] = (act && t0 > 0 && t0 - 1 < T) ? ld_keep4(h + base + (t0 - 1) * N) : f4(0.f);
#pragma unroll
    for (int k = 0; k < L; ++k) hv[k + 1] = (act && t0 + k < T) ? ld_keep4(h + base + (t0 + k) * N) : f4(0.f);
    mbar_wait(smem_u32(&s_bar), 0, &s_abort, status);

    // pass 1: composite of this thread's tokens from e_i = g_i c_i and b_i = a_{i+1}
    RevSeg G{f4(1.f), f4(0.f), false};
#pragma unroll
    for (int k = L - 1; k >= 0; --k) {
        const int64_t t = t0 + k;
        if (t >= T) continue;
        const int r = w * L + k;
        const float4 ev = srow(sg, r, lane) * srow(sc, r, lane);
        const float4 bv = t + 1 < T ? srow(sa, r + 1, lane) : f4(0.f);
        const bool end = (t == T - 1) || (TRUNC && (t + 1) % W == 0);
        if (end) G = RevSeg{bv, ev, true};
        else G = RevSeg{bv * G.Q, fma4(bv, G.S, ev), G.cl};
    }
    sQ[w][lane] = G.Q;
    sS[w][lane] = G.S;
    if (lane == 0) sCl[w] = G.cl;
    __syncthreads();

    // composite of the warps after this one and, in warp 0, the chunk aggregate
    RevSeg post{f4(1.f), f4(0.f), false};
    for (int j = w + 1; j < SC_WARPS; ++j) post = rseg_then(post, RevSeg{sQ[j][lane], sS[j][lane], sCl[j]});
    RevSeg agg{sQ[0][lane], sS[0][lane], sCl[0]};
    const int64_t di = seq * nchunks + chunk, fb = seq * nchunks;
    if (w == 0) {
#pragma unroll
        for (int j = 1; j < SC_WARPS; ++j) agg = rseg_then(agg, RevSeg{sQ[j][lane], sS[j][lane], sCl[j]});
        // A closed aggregate is already the inclusive composite: publish it before looking
        // back.  The look-back still runs, for the tokens after the chunk's last block end.
        if (agg.cl) desc_publish(&d.inc0[di * 32 + lane], agg.Q, &d.inc1[di * 32 + lane], agg.S);
        else desc_publish(&d.agg0[di * 32 + lane], agg.Q, &d.agg1[di * 32 + lane], agg.S);
    }
    // D_c = g h and E = c h need no carry: store them now, so these writes overlap the
    // look-back (after warp 0's publish, whose fence would otherwise wait for them).  The
    // g rows then hold e = g c for pass 2, and the c rows are free.
    float pz[DZ ? L : 1];   // DZ: this lane's share of dz per token (the D_c c part here)
    if (act) {
#pragma unroll
        for (int k = 0; k < L; ++k) {
            const int64_t t = t0 + k;
            if (t >= T) break;
            const int r = w * L + k;
            const float4 gk = srow(sg, r, lane), ck = srow(sc, r, lane);
            st4(Dc + base + t * N, gk * hv[k + 1]);
            st4(E + base + t * N, ck * hv[k + 1]);
            if (DZ) pz[k] = dot4(as_stored<TD>(gk * hv[k + 1]), ck);
            *reinterpret_cast<float4 *>(sg + r * SC_SLICE + lane * 4) = gk * ck;
        }
    }
    __syncthreads();   // sQ/sS/sCl now serve as look-back scratch
    // truncated mode: R at the window end of token t (row t + W - 1, the same local row)
    // lands in the c rows while the look-back runs
    if (TRUNC && threadIdx.x == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(smem_u32(&s_bar), uint32_t(TT) * SC_SLICE * 4u);
        tma_load_2d(smem_u32(sc), &mp.m[3], slice * SC_SLICE, int(b * T + c0 + W - 1), smem_u32(&s_bar));
    }
    RevSeg carry{f4(0.f), f4(0.f), true};
    if (chunk + 1 < nchunks) {
        carry = cta_lookback<RevSeg>(
            chunk + 1, 1, nchunks - 1 - chunk, RevSeg{f4(1.f), f4(0.f), false},
            [&](int64_t p, RevSeg &ag, bool &aok, RevSeg &ic, bool &iok) {
                const DescRead A = desc_read(&d.agg0[(fb + p) * 32 + lane], &d.agg1[(fb + p) * 32 + lane]);
                const DescRead I = desc_read(&d.inc0[(fb + p) * 32 + lane], &d.inc1[(fb + p) * 32 + lane]);
                ag = RevSeg{A.a, A.b, false};
                aok = A.ok;
                ic = RevSeg{I.a, I.b, true};
                iok = I.ok;
            },
            [](const RevSeg &acc, const RevSeg &g) { return rseg_then(acc, g); },
            RevSeg{f4(0.f), f4(0.f), true}, status, sQ, sS, sCl, s_ctl, w, lane);
    }
    if (w == 0) {
        if (!agg.cl) {
            const RevSeg inc = rseg_then(agg, carry);
            desc_publish(&d.inc0[di * 32 + lane], inc.Q, &d.inc1[di * 32 + lane], inc.S);
        }
        sCQ[lane] = carry.Q;
        sCS[lane] = carry.S;
    }
    __syncthreads();

    // composite of everything after this warp's tokens, then pass 2 backwards
    G = rseg_then(post, RevSeg{sCQ[lane], sCS[lane], true});
    if (TRUNC) mbar_wait(smem_u32(&s_bar), 1, &s_abort, status);
    const float4 bav = (DZ && act) ? *reinterpret_cast<const float4 *>(b_a + ch) : f4(0.f);
    static_assert(!DZ || L <= 8, "the row dots are summed eight tokens at a time");
    float vz[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = L - 1; k >= 0; --k) {
        const int64_t t = t0 + k;
        if (t >= T) continue;
        const int r = w * L + k;
        const float4 ak = srow(sa, r, lane);
        const float4 bk = t + 1 < T ? srow(sa, r + 1, lane) : f4(0.f);
        const float4 ek = srow(sg, r, lane);   // e = g c (written after pass 1)
        const bool end = (t == T - 1) || (TRUNC && (t + 1) % W == 0);
        if (end) G = RevSeg{bk, ek, true};
        else G = RevSeg{bk * G.Q, fma4(bk, G.S, ek), true};
        float4 mu = G.S;
        if (TRUNC && t % W != 0 && (t / W + 1) * W < T) {
            // the window ends at min(t + W - 1, T - 1); past the sequence end the staged row
            // is not this sequence's, so the last row is read directly
            const float4 rk = t + W - 1 <= T - 1 ? srow(sc, r, lane)
                                                 : (act ? ld_keep4(R + base + (T - 1) * N) : f4(0.f));
            mu = fma4(G.Q, rk, G.S);
        }
        const float4 dak = mu * hv[k] * ak * (f4(1.f) - ak);
        if (act) {
            st4(Du + base + t * N, mu);
            st4(Da + base + t * N, dak);
        }
        if (DZ && act) {
            const float4 za = make_float4(gate_z(ak.x, bav.x), gate_z(ak.y, bav.y), gate_z(ak.z, bav.z),
                                          gate_z(ak.w, bav.w));
            const float4 uk = hv[k + 1] - ak * hv[k];
            vz[k & 7] = pz[k] + dot4(as_stored<TD>(dak), za) + dot4(as_stored<TD>(mu), uk);
        }
    }
    if (DZ) {
        const float tot = warp_sum8(vz, lane);
        const int k = warp_sum8_index(lane);
        if ((lane & 3) == 0 && k < L && t0 + k < T) dz[(b * T + t0 + k) * nslices + slice] = tot;
    }
}

// ============================================================================ truncated adjoint in one pass
// The truncated adjoint in one reverse pass, for windows that are whole chunks
// (W % (8 L) == 0; blocks of W tokens then start at chunk starts).  With blocks of W tokens
// and s the start of the block after token i's, mu^W_i = S_i + Q_i R(i + W - 1), where R is
// the forward scan restarted at every block start (see the reverse scan above).  R is never
// scanned in a pass of its own:
//   * every chunk scans e = g c forward over its own rows only and stores these chunk-local
//     values R_loc (restarted at a block start, so a block's first chunk is closed), then
//     publishes the chunk's forward aggregate;
//   * the chunk that starts a block -- in reverse order the last of its block to run --
//     folds its block's aggregates into inclusive forward prefixes F and publishes them;
//   * a chunk of the block before reads the one prefix X = F of the chunk preceding its
//     window ends and gets R(m) = Sigma_X + Pi_X R_loc(m) from the stored local values, which
//     TMA brings into the freed c rows while its look-back runs.
// Chunks run block by block from the last, each block's chunks in reverse (one ticket each;
// trunc_order below), so every wait is on a CTA with an earlier ticket: the block's other
// chunks (aggregates), the block after's first chunk (prefixes).  Writers fence before they publish and readers after
// they observe, so the stored R_loc rows are visible to the TMA that reads them.  HBM sees
// the bytes of the full reverse scan plus the R_loc round trip, which mostly stays in L2.

// Wait (bounded) until a forward descriptor slot of this lane is published; returns it.
__device__ __forceinline__ FwdSeg wait_fdesc(const float4 *p0, const float4 *p1, unsigned *status) {
    for (int it = 0; it < SPIN_LIMIT; ++it) {
        const DescRead d = desc_read(p0, p1);
        if (__all_sync(0xffffffffu, d.ok)) return FwdSeg{d.a, d.b, false};
        if (it > 8) __nanosleep(64);
        if ((it & 255) == 255 && *reinterpret_cast<volatile unsigned *>(status) != 0u) break;
    }
    record_timeout(status);
    return FwdSeg{f4(1.f), f4(0.f), false};
}

// The same for n <= NB consecutive chunks' slots (p0, p1 of the first; a chunk's slots are 32
// float4 apart): all loads of a poll in flight at once, so a batch costs one L2 round trip.
// Ticket order: blocks of CB chunks from the last block back, and within a block each
// sequence's chunks in reverse, one sequence after the other (the last block may be short).
// The chunks of block k - 1 wait for the prefixes that block k's first chunk -- the last of
// its block and sequence to run -- folds; with several sequences the other sequences' chunks
// of block k run in between, so the fold is usually published before it is needed.  Every
// wait is still on an earlier ticket: a chunk's successors in its block and sequence, and
// the folds of later blocks of its sequence.
__device__ __forceinline__ void trunc_order(int64_t tk, int64_t nseq, int64_t nchunks, int64_t CB, int64_t &chunk,
                                            int64_t &seq) {
    const int64_t nblk = (nchunks + CB - 1) / CB, tail = nchunks - (nblk - 1) * CB;
    if (tk < nseq * tail) {
        seq = tk / tail;
        chunk = nchunks - 1 - tk % tail;
    } else {
        const int64_t u = tk - nseq * tail, g = u / (nseq * CB), r = u % (nseq * CB);
        seq = r / CB;
        chunk = (nblk - 2 - g) * CB + CB - 1 - r % CB;
    }
}

template <int NB>
__device__ __forceinline__ void wait_fdesc_n(const float4 *p0, const float4 *p1, int n, FwdSeg (&out)[NB],
                                             unsigned *status) {
    for (int it = 0; it < SPIN_LIMIT; ++it) {
        DescRead d[NB];
        bool ok = true;
#pragma unroll
        for (int u = 0; u < NB; ++u)
            if (u < n) {
                d[u] = desc_read(p0 + u * 32, p1 + u * 32);
                ok = ok && d[u].ok;
            }
        if (__all_sync(0xffffffffu, ok)) {
#pragma unroll
            for (int u = 0; u < NB; ++u) out[u] = u < n ? FwdSeg{d[u].a, d[u].b, false} : FwdSeg{f4(1.f), f4(0.f), false};
            return;
        }
        if (it > 8) __nanosleep(64);
        if ((it & 255) == 255 && *reinterpret_cast<volatile unsigned *>(status) != 0u) break;
    }
    record_timeout(status);
#pragma unroll
    for (int u = 0; u < NB; ++u) out[u] = FwdSeg{f4(1.f), f4(0.f), false};
}

template <int L, typename TD, bool DZ>
__global__ void __launch_bounds__(256, (L <= 4 ? 3 : 2)) k_trunc_scan(const __grid_constant__ ScanMaps mp, const float *__restrict__ h,
                                                      float *__restrict__ Rl, TD *__restrict__ Da, TD *__restrict__ Du,
                                                      TD *__restrict__ Dc, TD *__restrict__ E, int64_t T, int N,
                                                      int nslices, int64_t nseq, int64_t nchunks, int64_t W,
                                                      ScanWs dM, ScanWs dF, unsigned *status,
                                                      const float *__restrict__ b_a, float *__restrict__ dz) {
    constexpr int TT = SC_WARPS * L;
    extern __shared__ uint8_t sm_dyn[];
    float *sg = smem_1k(sm_dyn), *sc = sg + TT * SC_SLICE, *sa = sc + TT * SC_SLICE;
    __shared__ unsigned s_ticket;
    __shared__ uint64_t s_bar;
    __shared__ int s_abort;
    __shared__ float4 sX[SC_WARPS][32], sY[SC_WARPS][32], sC0[32], sC1[32];
    __shared__ bool sCl[SC_WARPS];
    __shared__ int s_ctl[SC_WARPS + 2];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t CB = W / TT;
    int64_t chunk, seq;
    trunc_order(chunk_ticket(dM, &s_ticket, &s_bar, &s_abort), nseq, nchunks, CB, chunk, seq);
    const int64_t b = seq / nslices;
    const int slice = int(seq % nslices), ch = slice * SC_SLICE + lane * 4;
    const bool act = ch < N;
    const int64_t c0 = chunk * TT, t0 = c0 + w * L;
    const int64_t base = b * T * N + ch;
    const int64_t di = seq * nchunks + chunk, fb = seq * nchunks;
    const int64_t blk = c0 / W;
    const bool first_of_block = c0 % W == 0;
    {
        float *dst[3] = {sg, sc, sa};
        const int rows[3] = {TT, TT, TT + 1};
        stage_chunk(mp, 3, dst, rows, slice * SC_SLICE, b * T + c0, &s_bar);
    }
    float4 hv[L + 1];
    hv[0] = (act && t0 > 0 && t0 - 1 < T) ? ld_keep4(h + base + (t0 - 1) * N) : f4(0.f);
#pragma unroll
    for (int k = 0; k < L; ++k) hv[k + 1] = (act && t0 + k < T) ? ld_keep4(h + base + (t0 + k) * N) : f4(0.f);
    mbar_wait(smem_u32(&s_bar), 0, &s_abort, status);

    // ---------------------------------------------------------------- forward, chunk-local
    // R_loc of this chunk's rows and the chunk's forward aggregate (blocks after the first
    // only: R of block 0 is never read)
    if (blk > 0) {
        FwdSeg G{f4(1.f), f4(0.f), false};
#pragma unroll
        for (int k = 0; k < L; ++k) {
            const int64_t t = t0 + k;
            if (t >= T) break;
            const int r = w * L + k;
            const float4 ev = srow(sg, r, lane) * srow(sc, r, lane), av = srow(sa, r, lane);
            if (t % W == 0) G = FwdSeg{f4(1.f), ev, true};
            else G = FwdSeg{G.P * av, fma4(G.P * av, ev, G.S), G.cl};
        }
        sX[w][lane] = G.P;
        sY[w][lane] = G.S;
        if (lane == 0) sCl[w] = G.cl;
        __syncthreads();
        FwdSeg pre{f4(1.f), f4(0.f), true};   // the chunk start: nothing before it
        for (int j = 0; j < w; ++j) pre = fseg_then(pre, FwdSeg{sX[j][lane], sY[j][lane], sCl[j]});
        FwdSeg agg{f4(1.f), f4(0.f), true};
        if (w == 0)
            for (int j = 0; j < SC_WARPS; ++j) agg = fseg_then(agg, FwdSeg{sX[j][lane], sY[j][lane], sCl[j]});
        G = pre;
#pragma unroll
        for (int k = 0; k < L; ++k) {
            const int64_t t = t0 + k;
            if (t >= T) break;
            const int r = w * L + k;
            const float4 ev = srow(sg, r, lane) * srow(sc, r, lane), av = srow(sa, r, lane);
            if (t % W == 0) G = FwdSeg{f4(1.f), ev, true};
            else G = FwdSeg{G.P * av, fma4(G.P * av, ev, G.S), G.cl};
            if (act) st4(Rl + base + t * N, G.S);   // kept in L2: the block before reads it soon
        }
        __syncthreads();   // every R_loc row stored (and sX/sY free again)
        if (w == 0) {
            __threadfence();
            desc_publish(&dF.agg0[di * 32 + lane], agg.P, &dF.agg1[di * 32 + lane], agg.S);
        }
        // the block's first chunk runs last of its block: fold the block's aggregates into the
        // inclusive prefixes the block before reads; warp j folds chunks [j q, (j + 1) q)
        if (first_of_block) {
            const int64_t cb = (c0 + W <= T ? W : T - c0 + TT - 1) / TT;   // chunks in this block
            const int64_t q = (cb + SC_WARPS - 1) / SC_WARPS, j0 = w * q, j1 = j0 + q < cb ? j0 + q : cb;
            // FOLD_NB aggregates a poll: the fold and the publication each take about q / FOLD_NB
            // L2 round trips (the block before waits on them)
            constexpr int FOLD_NB = 4;
            FwdSeg part{f4(1.f), f4(0.f), false};
            for (int64_t j = j0; j < j1; j += FOLD_NB) {
                const int64_t cj = fb + chunk + j;
                FwdSeg a_j[FOLD_NB];
                wait_fdesc_n<FOLD_NB>(&dF.agg0[cj * 32 + lane], &dF.agg1[cj * 32 + lane], int(j1 - j), a_j, status);
#pragma unroll
                for (int u = 0; u < FOLD_NB; ++u) part = fseg_then(part, a_j[u]);   // identity past j1
            }
            sX[w][lane] = part.P;
            sY[w][lane] = part.S;
            __syncthreads();
            FwdSeg run{f4(1.f), f4(0.f), true};   // the block start
            for (int j = 0; j < w; ++j) run = fseg_then(run, FwdSeg{sX[j][lane], sY[j][lane], false});
            __threadfence();   // every aggregate observed before any prefix is published
            for (int64_t j = j0; j < j1; j += FOLD_NB) {
                const int64_t cj = fb + chunk + j;
                DescRead d[FOLD_NB];
#pragma unroll
                for (int u = 0; u < FOLD_NB; ++u)
                    if (j + u < j1) d[u] = desc_read(&dF.agg0[(cj + u) * 32 + lane], &dF.agg1[(cj + u) * 32 + lane]);
#pragma unroll
                for (int u = 0; u < FOLD_NB; ++u)
                    if (j + u < j1) {
                        run = fseg_then(run, FwdSeg{d[u].a, d[u].b, false});
                        desc_publish(&dF.inc0[(cj + u) * 32 + lane], run.P, &dF.inc1[(cj + u) * 32 + lane], run.S);
                    }
            }
            __syncthreads();   // sX/sY free again
        }
    }

    // ---------------------------------------------------------------- reverse (restarted at block ends)
    RevSeg G{f4(1.f), f4(0.f), false};
#pragma unroll
    for (int k = L - 1; k >= 0; --k) {
        const int64_t t = t0 + k;
        if (t >= T) continue;
        const int r = w * L + k;
        const float4 ev = srow(sg, r, lane) * srow(sc, r, lane);
        const float4 bv = t + 1 < T ? srow(sa, r + 1, lane) : f4(0.f);
        const bool end = (t == T - 1) || ((t + 1) % W == 0);
        if (end) G = RevSeg{bv, ev, true};
        else G = RevSeg{bv * G.Q, fma4(bv, G.S, ev), G.cl};
    }
    sX[w][lane] = G.Q;
    sY[w][lane] = G.S;
    if (lane == 0) sCl[w] = G.cl;
    __syncthreads();
    RevSeg post{f4(1.f), f4(0.f), false};
    for (int j = w + 1; j < SC_WARPS; ++j) post = rseg_then(post, RevSeg{sX[j][lane], sY[j][lane], sCl[j]});
    RevSeg agg{sX[0][lane], sY[0][lane], sCl[0]};
    if (w == 0) {
#pragma unroll
        for (int j = 1; j < SC_WARPS; ++j) agg = rseg_then(agg, RevSeg{sX[j][lane], sY[j][lane], sCl[j]});
        if (agg.cl) desc_publish(&dM.inc0[di * 32 + lane], agg.Q, &dM.inc1[di * 32 + lane], agg.S);
        else desc_publish(&dM.agg0[di * 32 + lane], agg.Q, &dM.agg1[di * 32 + lane], agg.S);
    }
    float pz[DZ ? L : 1];
    if (act) {
#pragma unroll
        for (int k = 0; k < L; ++k) {
            const int64_t t = t0 + k;
            if (t >= T) break;
            const int r = w * L + k;
            const float4 gk = srow(sg, r, lane), ck = srow(sc, r, lane);
            st4(Dc + base + t * N, gk * hv[k + 1]);
            st4(E + base + t * N, ck * hv[k + 1]);
            if (DZ) pz[k] = dot4(as_stored<TD>(gk * hv[k + 1]), ck);
            *reinterpret_cast<float4 *>(sg + r * SC_SLICE + lane * 4) = gk * ck;
        }
    }
    __syncthreads();
    // The window ends m = min(t + W - 1, T - 1) of this chunk's tokens lie in the next block,
    // in chunk cx = chunk + CB - 1 (only m = c0 + W - 1, the end of cx), in chunk cx + 1, or
    // at T - 1 in the last chunk cl.  R(m) is then the inclusive prefix of cx (end of cx),
    // that of cl (m = T - 1), or, inside cx + 1, the prefix of cx composed with the stored
    // local value (identity prefix when cx + 1 starts the block, i.e. this chunk starts its
    // own).  Those rows come by TMA into the freed c rows while the look-back runs, once cx + 1's
    // prefix -- published after every R_loc row of the block was stored -- is seen.
    const bool need_r = (blk + 1) * W < T;
    const int64_t cl = nchunks - 1, cx = chunk + CB - 1;
    const bool use_rows = need_r && c0 + W + 1 < T;                       // some m inside cx + 1
    const bool use_x = need_r && !first_of_block && c0 + W < T;           // prefix of cx needed
    const bool use_end = need_r && c0 + TT + W - 2 >= T - 1;              // some m clamped to T - 1
    if (use_rows && w == 0) {
        (void)wait_fdesc(&dF.inc0[(fb + cx + 1) * 32 + lane], &dF.inc1[(fb + cx + 1) * 32 + lane], status);
        if (lane == 0) {
            __threadfence();
            fence_proxy_async_global();   // the rows were stored through the generic proxy
            fence_proxy_async_smem();     // the c rows were read through it
            mbar_arrive_expect_tx(smem_u32(&s_bar), uint32_t(TT) * SC_SLICE * 4u);
            tma_load_2d(smem_u32(sc), &mp.m[3], slice * SC_SLICE, int(b * T + c0 + W - 1), smem_u32(&s_bar));
        }
        __syncwarp();
    }
    RevSeg carry{f4(0.f), f4(0.f), true};
    // a block's last chunk ends closed (W is whole chunks): nothing after it counts
    if (chunk + 1 < nchunks && (c0 + TT) % W != 0) {
        carry = cta_lookback<RevSeg>(
            chunk + 1, 1, nchunks - 1 - chunk, RevSeg{f4(1.f), f4(0.f), false},
            [&](int64_t p, RevSeg &ag, bool &aok, RevSeg &ic, bool &iok) {
                const DescRead A = desc_read(&dM.agg0[(fb + p) * 32 + lane], &dM.agg1[(fb + p) * 32 + lane]);
                const DescRead I = desc_read(&dM.inc0[(fb + p) * 32 + lane], &dM.inc1[(fb + p) * 32 + lane]);
                ag = RevSeg{A.a, A.b, false};
                aok = A.ok;
                ic = RevSeg{I.a, I.b, true};
                iok = I.ok;
            },
            [](const RevSeg &acc, const RevSeg &g) { return rseg_then(acc, g); },
            RevSeg{f4(0.f), f4(0.f), true}, status, sX, sY, sCl, s_ctl, w, lane);
    }
    if (w == 0) {
        if (!agg.cl) {
            const RevSeg inc = rseg_then(agg, carry);
            desc_publish(&dM.inc0[di * 32 + lane], inc.Q, &dM.inc1[di * 32 + lane], inc.S);
        }
        sC0[lane] = carry.Q;
        sC1[lane] = carry.S;
    }
    __syncthreads();
    // this lane's parts of the prefixes it reads (bounded waits on validated descriptors)
    FwdSeg X{f4(1.f), f4(0.f), true}, XE{f4(1.f), f4(0.f), true};
    if (use_x) X = wait_fdesc(&dF.inc0[(fb + cx) * 32 + lane], &dF.inc1[(fb + cx) * 32 + lane], status);
    if (use_end) XE = wait_fdesc(&dF.inc0[(fb + cl) * 32 + lane], &dF.inc1[(fb + cl) * 32 + lane], status);
    G = rseg_then(post, RevSeg{sC0[lane], sC1[lane], true});
    if (use_rows) mbar_wait(smem_u32(&s_bar), 1, &s_abort, status);
    const float4 bav = (DZ && act) ? *reinterpret_cast<const float4 *>(b_a + ch) : f4(0.f);
    static_assert(!DZ || L <= 8, "the row dots are summed eight tokens at a time");
    float vz[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int64_t xend = (cx + 1) * TT;   // window ends before this row are the end of chunk cx
#pragma unroll
    for (int k = L - 1; k >= 0; --k) {
        const int64_t t = t0 + k;
        if (t >= T) continue;
        const int r = w * L + k;
        const float4 ak = srow(sa, r, lane);
        const float4 bk = t + 1 < T ? srow(sa, r + 1, lane) : f4(0.f);
        const float4 ek = srow(sg, r, lane);
        const bool end = (t == T - 1) || ((t + 1) % W == 0);
        if (end) G = RevSeg{bk, ek, true};
        else G = RevSeg{bk * G.Q, fma4(bk, G.S, ek), true};
        float4 mu = G.S;
        if (t % W != 0 && need_r) {
            const int64_t m = t + W - 1 <= T - 1 ? t + W - 1 : T - 1;
            const float4 rk = m == T - 1 ? XE.S
                              : m < xend  ? X.S
                                          : fma4(X.P, srow(sc, int(m - (c0 + W - 1)), lane), X.S);
            mu = fma4(G.Q, rk, G.S);
        }
        const float4 dak = mu * hv[k] * ak * (f4(1.f) - ak);
        if (act) {
            st4(Du + base + t * N, mu);
            st4(Da + base + t * N, dak);
        }
        if (DZ && act) {
            const float4 za = make_float4(gate_z(ak.x, bav.x), gate_z(ak.y, bav.y), gate_z(ak.z, bav.z),
                                          gate_z(ak.w, bav.w));
            const float4 uk = hv[k + 1] - ak * hv[k];
            vz[k & 7] = pz[k] + dot4(as_stored<TD>(dak), za) + dot4(as_stored<TD>(mu), uk);
        }
    }
    if (DZ) {
        const float tot = warp_sum8(vz, lane);
        const int k = warp_sum8_index(lane);
        if ((lane & 3) == 0 && k < L && t0 + k < T) dz[(b * T + t0 + k) * nslices + slice] = tot;
    }
}

// ============================================================================ launchers
// Maps of the staged arrays ([B*T rows, N cols] fp32, boxes of 128 channels x rows[i]).
static bool scan_maps(ScanMaps &mp, int n, const float *const *arr, const int *rows, int64_t B, int64_t T, int N) {
    memset(&mp, 0, sizeof(mp));
    for (int i = 0; i < n; ++i)
        if (!tmap_rows_f32(&mp.m[i], arr[i], uint64_t(N), uint64_t(B * T), uint64_t(N) * 4, SC_SLICE, uint32_t(rows[i])))
            return false;
    return true;
}
static size_t staged_bytes(int total_rows) { return size_t(total_rows) * SC_SLICE * 4 + 1024; }

template <class K>
static cudaError_t set_smem(K kern, size_t smem) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

cudaError_t launch_fwd_scan(const float *a, const float *u, float *h, int64_t B, int64_t T, int N,
                            void *scan_ws, unsigned *status, cudaStream_t st, bool withhold_first,
                            const float *c, __nv_bfloat16 *ch) {
    constexpr int L = SC_FWD_L, TT = SC_WARPS * L;
    const int nslices = int(cdiv(N, SC_SLICE));
    const int64_t nseq = B * nslices, nchunks = cdiv(T, TT);
    if (withhold_first && (nseq != 1 || nchunks < 2)) return cudaErrorInvalidValue;
    ScanMaps mp;
    const float *arr[2] = {a, u};
    const int rows[2] = {TT, TT};
    if (!scan_maps(mp, 2, arr, rows, B, T, N)) return cudaErrorInvalidValue;
    ScanWs d = scan_ws_carve(scan_ws, nseq * nchunks);
    cudaError_t e = scan_ws_reset(scan_ws, nseq * nchunks, st);
    if (e != cudaSuccess) return e;
    // self test of the look-back's give-up path: the ticket starts one chunk ahead and the
    // grid is one chunk short, so chunk 0 never runs and never publishes, and every other
    // chunk's look-back waits for it until its limit
    if (withhold_first && (e = cudaMemsetAsync(d.ticket, 0, sizeof(unsigned), st)) != cudaSuccess) return e;
    const size_t smem = staged_bytes(2 * TT);
    const unsigned grid = unsigned(nseq * nchunks - (withhold_first ? 1 : 0));
    if (c && ch) {
        if ((e = set_smem(k_fwd_scan<L, true>, smem)) != cudaSuccess) return e;
        k_fwd_scan<L, true><<<grid, 256, smem, st>>>(mp, h, c, ch, T, N, nslices, nseq, nchunks, d, status);
    } else {
        if ((e = set_smem(k_fwd_scan<L, false>, smem)) != cudaSuccess) return e;
        k_fwd_scan<L, false><<<grid, 256, smem, st>>>(mp, h, nullptr, nullptr, T, N, nslices, nseq, nchunks, d, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_win_scan(const float *g, const float *c, const float *a, float *R, int64_t B,
                            int64_t T, int N, int64_t W, void *scan_ws, unsigned *status, cudaStream_t st) {
    constexpr int L = SC_BWD_L, TT = SC_WARPS * L;
    const int nslices = int(cdiv(N, SC_SLICE));
    const int64_t nseq = B * nslices, nchunks = cdiv(T, TT);
    ScanMaps mp;
    const float *arr[3] = {g, c, a};
    const int rows[3] = {TT, TT, TT};
    if (!scan_maps(mp, 3, arr, rows, B, T, N)) return cudaErrorInvalidValue;
    ScanWs d = scan_ws_carve(scan_ws, nseq * nchunks);
    cudaError_t e = scan_ws_reset(scan_ws, nseq * nchunks, st);
    if (e != cudaSuccess) return e;
    const size_t smem = staged_bytes(3 * TT);
    if ((e = set_smem(k_win_scan<L>, smem)) != cudaSuccess) return e;
    k_win_scan<L><<<unsigned(nseq * nchunks), 256, smem, st>>>(mp, R, T, N, nslices, nseq, nchunks, W, d, status);
    return cudaGetLastError();
}

// Scan workspace of the one-pass truncated adjoint: two descriptor sets, laid out
// [ticket, reverse descriptors | ticket (unused), forward descriptors].
static int64_t trunc_chunks(int64_t B, int64_t T, int N) {
    return B * cdiv(N, SC_SLICE) * cdiv(T, SC_WARPS * SC_TRUNC_L);
}
static size_t trunc_desc_bytes(int64_t n) { return 256 + 4 * size_t(n) * 32 * sizeof(float4); }
size_t trunc_ws_bytes(int64_t B, int64_t T, int N) { return 2 * trunc_desc_bytes(trunc_chunks(B, T, N)); }
bool trunc_one_launch(int64_t T, int64_t W) { return W > 0 && W < T && W % (SC_WARPS * SC_TRUNC_L) == 0; }

cudaError_t launch_trunc_scan(const float *g, const float *c, const float *a, const float *h, float *R, void *D_a,
                              void *D_u, void *D_c, void *E, bool d_bf16, int64_t B, int64_t T, int N, int64_t W,
                              void *ws, unsigned *status, cudaStream_t st, const float *b_a, float *dz) {
    constexpr int L = SC_TRUNC_L, TT = SC_WARPS * L;
    if (!trunc_one_launch(T, W)) return cudaErrorInvalidValue;
    const int nslices = int(cdiv(N, SC_SLICE));
    const int64_t nseq = B * nslices, nchunks = cdiv(T, TT), n = nseq * nchunks;
    ScanMaps mp;
    const float *arr[4] = {g, c, a, R};
    const int rows[4] = {TT, TT, TT + 1, TT};
    if (!scan_maps(mp, 4, arr, rows, B, T, N)) return cudaErrorInvalidValue;
    char *p = static_cast<char *>(ws);
    const ScanWs dM = scan_ws_carve(p, n), dF = scan_ws_carve(p + trunc_desc_bytes(n), n);
    // every descriptor word unset, the ticket at 0xFFFFFFFF: one memset
    cudaError_t e = cudaMemsetAsync(ws, 0xFF, 2 * trunc_desc_bytes(n), st);
    if (e != cudaSuccess) return e;
    const unsigned grid = unsigned(n);
    const size_t smem = staged_bytes(3 * TT + 1);
#define ADJ_TRUNC(TDT, DZO)                                                                                      \
    do {                                                                                                         \
        if ((e = set_smem(k_trunc_scan<L, TDT, DZO>, smem)) != cudaSuccess) return e;                            \
        k_trunc_scan<L, TDT, DZO><<<grid, 256, smem, st>>>(mp, h, R, static_cast<TDT *>(D_a), static_cast<TDT *>(D_u), \
                                                          static_cast<TDT *>(D_c), static_cast<TDT *>(E), T, N,       \
                                                          nslices, nseq, nchunks, W, dM, dF, status, b_a, dz);        \
    } while (0)
    if (d_bf16) {
        if (dz) ADJ_TRUNC(__nv_bfloat16, true);
        else ADJ_TRUNC(__nv_bfloat16, false);
    } else {
        if (dz) ADJ_TRUNC(float, true);
        else ADJ_TRUNC(float, false);
    }
#undef ADJ_TRUNC
    return cudaGetLastError();
}

cudaError_t launch_bwd_scan(const float *g, const float *c, const float *a, const float *h, const float *R,
                            void *D_a, void *D_u, void *D_c, void *E, bool d_bf16, int64_t B, int64_t T, int N,
                            int64_t W, void *scan_ws, unsigned *status, cudaStream_t st, const float *b_a,
                            float *dz) {
    constexpr int L = SC_BWD_L, TT = SC_WARPS * L;
    const int nslices = int(cdiv(N, SC_SLICE));
    const int64_t nseq = B * nslices, nchunks = cdiv(T, TT);
    const bool trunc = W > 0 && W < T;
    ScanMaps mp;
    const float *arr[4] = {g, c, a, R};
    const int rows[4] = {TT, TT, TT + 1, TT};
    if (!scan_maps(mp, trunc ? 4 : 3, arr, rows, B, T, N)) return cudaErrorInvalidValue;
    ScanWs d = scan_ws_carve(scan_ws, nseq * nchunks);
    cudaError_t e = scan_ws_reset(scan_ws, nseq * nchunks, st);
    if (e != cudaSuccess) return e;
    const unsigned grid = unsigned(nseq * nchunks);
    const size_t smem = staged_bytes(3 * TT + 1);
#define ADJ_BWD(TR, TDT, DZO)                                                                                     \
    do {                                                                                                          \
        if ((e = set_smem(k_bwd_scan<L, TR, TDT, DZO>, smem)) != cudaSuccess) return e;                           \
        k_bwd_scan<L, TR, TDT, DZO><<<grid, 256, smem, st>>>(mp, h, R, static_cast<TDT *>(D_a),                   \
                                                             static_cast<TDT *>(D_u), static_cast<TDT *>(D_c),    \
                                                             static_cast<TDT *>(E), T, N, nslices, nseq, nchunks, \
                                                             trunc ? W : T, d, status, b_a, dz);                  \
    } while (0)
#define ADJ_BWD_DZ(TR, TDT)               \
    do {                                  \
        if (dz) ADJ_BWD(TR, TDT, true);   \
        else ADJ_BWD(TR, TDT, false);     \
    } while (0)
    if (d_bf16) {
        if (trunc) ADJ_BWD_DZ(true, __nv_bfloat16);
        else ADJ_BWD_DZ(false, __nv_bfloat16);
    } else {
        if (trunc) ADJ_BWD_DZ(true, float);
        else ADJ_BWD_DZ(false, float);
    }
#undef ADJ_BWD_DZ
#undef ADJ_BWD
    return cudaGetLastError();
}

}  // namespace adj
