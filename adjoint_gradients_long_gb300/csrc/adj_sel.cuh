// adj_sel.cuh -- launchers of the general selective layer's scans (adj_sel.cu).  Not part
// of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace adj {

constexpr int SEL_NT = 8;          // states a thread owns
constexpr int SEL_TT_MAX = 256;    // tokens a chunk (full adjoint)
constexpr int SEL_TT_MIN = 16;     // smallest chunk; truncation windows are multiples of it

// chunk length for T tokens and window W (W <= 0 or W >= T: full): the largest power of two
// up to SEL_TT_MAX that divides W, so that blocks of W tokens start at chunk starts
int sel_chunk(int64_t T, int64_t W);
bool sel_window_ok(int64_t T, int64_t W);
// CTAs across the channels: ceil(P / (256 / (NS / 8)))
int sel_slices(int P, int NS);

// Scratch of the reverse pass, carved from the caller's workspace:
//   aggX, aggY  [B, nchunks, P, NS]   reverse-scan chunk aggregates, then carries
//   winX, winY  [B, nchunks, P, NS]   window-scan aggregates/carries (truncated only)
//   R           [B, T, P, NS]         window sums R (truncated only)
//   bc          [B*T, slices, 2 NS]   per-CTA partial sums of dB and dC
//   dAp         [B*nchunks, P, NS]    per-chunk partial sums of dA
struct SelBwdWs {
    float *aggX, *aggY, *winX, *winY, *R, *bc, *dAp;
};

// The reverse pass's input path (a layer of a stack that reads the normalised residual
// stream; all null for a lone layer):
//   r       [B*T]              the rms of the layer's input stream
//   gadd    [B,T,P]   out      gy + dt sum_n mu^W B / r (the input term's share of the
//                              cotangent below, before the normalisation's row term)
//   rowdot  [B*T, slices + 1]  out  per-CTA partial sums of xhat . dxhat (the projection's
//                              share as dz . z)
struct SelInp {
    const float *r;
    float *gadd, *rowdot;
};

// h [B,T,P,NS], y [B,T,P] from z = xhat W_in (without b_dt) [B,T,P+2NS]; y = xres + sum_n C h
// (xres null: xhat); aggX/aggY: two [B, nchunks, P, NS] scratch arrays.
cudaError_t launch_sel_fwd(const float *z, const void *x, bool x_bf16, const float *b_dt, const float *A, float *h,
                           float *y, const float *xres, float *aggX, float *aggY, int64_t B, int64_t T, int P, int NS,
                           cudaStream_t st);
// dz [B,T,P+2NS] (d_bf16: bf16) and dA [P,NS] for the cotangent gy [B,T,P]; W <= 0 or
// W >= T: full adjoint.  status: the workspace status word (a bounded wait for a bulk copy
// that gave up records the timeout there).
cudaError_t launch_sel_bwd(const float *z, const void *x, bool x_bf16, const float *gy, const float *h,
                           const float *b_dt, const float *A, void *dz, bool d_bf16, float *dA, const SelBwdWs &w,
                           const SelInp &inp, int64_t B, int64_t T, int P, int NS, int64_t W, unsigned *status,
                           cudaStream_t st);
// part[blk][p] = sum of dz[:, p] over row block blk (nblk contiguous blocks of the rows)
cudaError_t launch_sel_colsum(const void *dz, bool d_bf16, int64_t rows, int P, int ld, int nblk, float *part,
                              cudaStream_t st);

}  // namespace adj
