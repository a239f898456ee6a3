// adj_internal.cuh -- helpers shared by the kernels of libadj.so (device side and
// launcher declarations).  Nothing here is part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/adj.h"

namespace adj {

// ---------------------------------------------------------------- status word
// Word 0 of the workspace: sticky device status; bit ADJ_ST_TIMEOUT is set by a
// bounded wait that gave up.  Word 1: the loss kernel's wrapping block ticket.  Words
// 2..63 are reserved.
constexpr unsigned ST_TIMEOUT = 1u;
constexpr size_t WS_HEADER = 256;

// Iteration limit of the scans' look-back (rounds, each one L2 round trip plus a short
// back-off): a wait that never ends gives up after a few seconds.
constexpr int SPIN_LIMIT = 1 << 22;

__device__ __forceinline__ void record_timeout(unsigned *status) {
    atomicOr(status, ST_TIMEOUT);
}

// ---------------------------------------------------------------- memory ops
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// L2-coherent loads/stores for look-back descriptors (never served from a stale L1 line).
__device__ __forceinline__ float4 ld_cg4(const float4 *p) { return __ldcg(p); }
__device__ __forceinline__ void st_cg4(float4 *p, float4 v) { __stcg(p, v); }

// streaming loads/stores of the big token-major arrays
__device__ __forceinline__ float4 ld_stream4(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ float4 ld_keep4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ void st_stream4(float *p, float4 v) { __stcs(reinterpret_cast<float4 *>(p), v); }

__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<unsigned *>(&lo);
    u.y = *reinterpret_cast<unsigned *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}

// ---------------------------------------------------------------- float4 arithmetic
__device__ __forceinline__ float4 f4(float s) { return make_float4(s, s, s, s); }
__device__ __forceinline__ float4 operator*(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
__device__ __forceinline__ float4 operator+(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ float4 operator-(float4 a, float4 b) { return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }
// a * b + c, one rounding per lane
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {
    return make_float4(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y), fmaf(a.z, b.z, c.z), fmaf(a.w, b.w, c.w));
}

// ---------------------------------------------------------------- launchers
struct ScanWs {               // look-back descriptors carved from the workspace
    unsigned *ticket;         // 1 counter
    float4 *agg0, *agg1;      // [nseq * nchunks * 32] chunk aggregates (2 components)
    float4 *inc0, *inc1;      // [nseq * nchunks * 32] inclusive prefixes
};

size_t scan_ws_bytes(int64_t B, int64_t T, int N);
ScanWs scan_ws_carve(void *base, int64_t nchunks_total);

// withhold_first (self test only, B * ceil(N/128) == 1): chunk 0 never runs, so every
// other chunk's look-back waits for it until its limit and records a timeout.
// c and ch (both or neither): also write ch = bf16(c . h) [B,T,N].
cudaError_t launch_fwd_scan(const float *a, const float *u, float *h, int64_t B, int64_t T, int N,
                            void *scan_ws, unsigned *status, cudaStream_t st, bool withhold_first = false,
                            const float *c = nullptr, __nv_bfloat16 *ch = nullptr);
cudaError_t launch_win_scan(const float *g, const float *c, const float *a, float *R, int64_t B,
                            int64_t T, int N, int64_t Tbar, void *scan_ws, unsigned *status,
                            cudaStream_t st);
// The truncated adjoint in one reverse pass (no separate window scan), for windows of whole
// scan chunks (trunc_one_launch); its scan workspace is trunc_ws_bytes.  R [B,T,N] is its
// scratch for the chunk-local window sums.
bool trunc_one_launch(int64_t T, int64_t W);
size_t trunc_ws_bytes(int64_t B, int64_t T, int N);
cudaError_t launch_trunc_scan(const float *g, const float *c, const float *a, const float *h, float *R, void *D_a,
                              void *D_u, void *D_c, void *E, bool d_bf16, int64_t B, int64_t T, int N, int64_t W,
                              void *ws, unsigned *status, cudaStream_t st, const float *b_a = nullptr,
                              float *dz = nullptr);
// dz (with b_a; both or neither): also the per-token, per-128-channel-slice sums
// [B*T, ceil(N/128)] of D_a z_a + D_u u + D_c c (the row dot xhat . dxhat of the layer input)
cudaError_t launch_bwd_scan(const float *g, const float *c, const float *a, const float *h,
                            const float *R, void *D_a, void *D_u, void *D_c, void *E, bool d_bf16,
                            int64_t B, int64_t T, int N, int64_t Tbar, void *scan_ws,
                            unsigned *status, cudaStream_t st, const float *b_a = nullptr, float *dz = nullptr);

// GEMM operands: strided, optionally split over up to three arrays.
struct GemmOperand {
    const void *p[3];    // up to three arrays split along K (A) or along Nc (B)
    const void *lo[3];   // pre-split operand: bf16 low parts of p (then p holds the bf16
                         // high parts, x = hi + lo); null otherwise
    int64_t blk;         // split size (K for A, Nc for B); >= the dimension if one array
    int64_t s_row;       // stride of the M (A) / Nc (B) index within one array
    int64_t s_k;         // stride of the K index
    bool bf16;           // element type: bf16 or fp32
    const float *mul;    // optional fp32 array multiplied elementwise (A only, same strides)
};

enum class Epi { ProjIn, Store, StoreAdd, Partial };

struct GemmEpilogue {
    Epi kind;
    float *out0, *out1, *out2;  // ProjIn: a, u, c [M,N]; Store/StoreAdd: out0 [M,ld]; Partial: out0 base
    void *out_x;                // Store/StoreAdd: optional bf16 copy of out0
    const void *add;            // StoreAdd: out0 = acc + add (fp32, or bf16 if add_bf16)
    bool add_bf16;
    const float *bias;          // ProjIn: b_a [N]
    int64_t ld;                 // row stride of out0/add/out_x
    int N;                      // ProjIn: width of each block
    bool interleave;            // ProjIn: product column chunk j (32 columns) is block j % 3,
                                // channels 32 (j / 3) ...; needs N % 32 == 0 (see prep_win)
    // Partial with a row-contiguous fp32 B converted by the producers: also the column sums
    // of B's first csum_n columns, csum [2 * splits][csum_n] (two partials a split).  The
    // launch reports whether it took them (csum_done); otherwise csum is left untouched.
    float *csum;
    int64_t csum_n;
    // StoreAdd through a normalised layer input xhat = y / r (nr non-null):
    //   out0[m,n] = add[m,n] + (acc - nx[m,n] * (sum_{s < nsl} ndz[m * nsl + s]) * inv_P) / nr[m]
    // with nx [M, ld] (bf16 if nx_bf16, else fp32), nr [M], ndz [M, nsl] fp32.
    const float *nr;
    const float *ndz;
    int nsl;
    const void *nx;
    bool nx_bf16;
    float inv_P;
};

// ProjIn output column n of the product -> block (0 a, 1 u, 2 c) and channel.
__host__ __device__ inline void projin_col(const GemmEpilogue &ep, int n, int &blk, int &ch) {
    if (ep.interleave) {
        const int j = n >> 5;
        blk = j % 3;
        ch = (j / 3) * 32 + (n & 31);
    } else {
        blk = n / ep.N;
        ch = n - blk * ep.N;
    }
}

// tcgen05 GEMM C[M,Nc] = A[M,K] B[K,Nc] with the operand and epilogue contracts above;
// split3: fp32-accurate hi/lo bf16 split, otherwise bf16 operands.
cudaError_t launch_gemm_tc(int64_t M, int64_t Nc, int64_t K, const GemmOperand &A, const GemmOperand &Bm,
                           const GemmEpilogue &ep, int splits, bool split3, unsigned *status, cudaStream_t st,
                           int *splits_used = nullptr, bool *csum_done = nullptr);

// W_in [P, 3N] with its columns interleaved in 32-column chunks (chunk j of the copy =
// columns 32 (j / 3) ... of block j % 3, so every wide output tile mixes the a, u and c
// blocks): fp32 weights -> bf16 hi and lo copies, bf16 weights -> a bf16 copy (lo null).
// With wo (fp32 [N, P]), the same launch also splits W_o into wo_hi and wo_lo.
cudaError_t launch_prep_win(const void *w, bool w_bf16, int P, int N, __nv_bfloat16 *hi, __nv_bfloat16 *lo,
                            cudaStream_t st, const float *wo = nullptr, __nv_bfloat16 *wo_hi = nullptr,
                            __nv_bfloat16 *wo_lo = nullptr);
// hi = bf16(w), lo = bf16(w - hi) for n fp32 values (operands of the split-precision GEMM)
cudaError_t launch_split_bf16(const float *w, int64_t n, __nv_bfloat16 *hi, __nv_bfloat16 *lo, cudaStream_t st);
// One array of partials to reduce: out[i] (+)= sum_{z < splits} part[z * 4 n4 + i] over
// i < 4 n4 (16-byte aligned; group and first, the array's first block, are filled in by
// the launcher).
struct RedSeg {
    const float *part;
    float *out;
    int64_t n4;
    int splits;
    int group;
    int64_t first;
};
struct RedArgs {
    RedSeg seg[3];
    int nseg;
    int accumulate;
};
// Reduces up to three arrays of partials in one launch, deterministically.
cudaError_t launch_reduce_partials(const RedSeg *segs, int nseg, int accumulate, cudaStream_t st);
// part[blk][n] = column sums of D over block blk's rows (nblk contiguous row ranges)
cudaError_t launch_colsum(const void *D, bool bf16, int64_t rows, int N, float *part, int nblk, cudaStream_t st);
cudaError_t launch_rms_norm(const float *y, void *xhat, bool xbf, float *r, int64_t rows, int P, float eps,
                            cudaStream_t st);
cudaError_t launch_rms_norm_bwd(const float *y, const float *r, const float *dx, const float *gy, float *gy_prev,
                                int64_t rows, int P, cudaStream_t st);
// ticket: a word of the workspace header (zero before the first call, back at zero after
// every launch)
cudaError_t launch_loss(const float *y, const float *target, float *gy, __nv_bfloat16 *gyx, int64_t count,
                        double *part, int nblk, unsigned *ticket, double *loss, cudaStream_t st);

}  // namespace adj
