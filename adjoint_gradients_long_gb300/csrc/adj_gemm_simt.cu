// adj_gemm_simt.cu -- fp32 SIMT tiled GEMM with fused prologue/epilogue for the
// projections of the adjoint-sharding path.  It reads operands of any stride and
// either storage type (fp32 or bf16) and accumulates in fp32.
//
// Roles ([AS] = review page "Adjoint sharding for very long context training of
// state space models"; model of [AS] Assumptions, Sec. 3.1):
//   proj_in    [a|u|c] = xhat W_in, a = sigmoid(. + b_a)      (epilogue ProjIn)
//   proj_out   y = xres + (c . h) W_o                          (A prologue c.h, StoreAdd)
//   cot_proj   g = gy W_o^T                                     (Store)
//   param      dW_in = xhat^T [D_a|D_u|D_c], dW_o = E^T gy      (split over tokens, Partial)
//   input_grad gy_prev = gy + [D_a|D_u|D_c] W_in^T              (StoreAdd)
#include "adj_internal.cuh"
#include "adj_epilogue.cuh"

namespace adj {

constexpr int GB_M = 64, GB_N = 64, GB_K = 16;

template <bool BF>
__device__ __forceinline__ float ld_elem(const void *p, int64_t i) {
    if (BF) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    return static_cast<const float *>(p)[i];
}

// A(m, k): arrays split along k
template <bool BF>
__device__ __forceinline__ float ld_A(const GemmOperand &A, int64_t m, int64_t k) {
    const int blk = int(k / A.blk);
    const int64_t i = m * A.s_row + (k - blk * A.blk) * A.s_k;
    float v = ld_elem<BF>(A.p[blk], i);
    if (A.mul) v *= A.mul[i];
    return v;
}
// B(k, n): arrays split along n
template <bool BF>
__device__ __forceinline__ float ld_B(const GemmOperand &Bm, int64_t k, int64_t n) {
    const int blk = int(n / Bm.blk);
    const int64_t i = (n - blk * Bm.blk) * Bm.s_row + k * Bm.s_k;
    return ld_elem<BF>(Bm.p[blk], i);
}

template <bool ABF, bool BBF>
__global__ void __launch_bounds__(256) k_gemm_simt(int64_t M, int64_t Nc, int64_t K, GemmOperand A,
                                                   GemmOperand Bm, GemmEpilogue ep, int64_t kper) {
    __shared__ float sA[GB_K][GB_M + 4];
    __shared__ float sB[GB_K][GB_N + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int64_t m0 = int64_t(blockIdx.y) * GB_M, n0 = int64_t(blockIdx.x) * GB_N;
    const int z = blockIdx.z;
    const int64_t kb = int64_t(z) * kper, ke = kb + kper < K ? kb + kper : K;
    const bool a_kfast = A.s_k == 1, b_nfast = Bm.s_row == 1;
    float acc[4][4] = {};
    for (int64_t k0 = kb; k0 < ke; k0 += GB_K) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = tid + r * 256;
            const int mi = a_kfast ? e / GB_K : e % GB_M, ki = a_kfast ? e % GB_K : e / GB_M;
            const int64_t m = m0 + mi, k = k0 + ki;
            sA[ki][mi] = (m < M && k < ke) ? ld_A<ABF>(A, m, k) : 0.f;
            const int ni = b_nfast ? e % GB_N : e / GB_K, kj = b_nfast ? e / GB_N : e % GB_K;
            const int64_t n = n0 + ni, kk = k0 + kj;
            sB[kj][ni] = (n < Nc && kk < ke) ? ld_B<BBF>(Bm, kk, n) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GB_K; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = sA[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = sB[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
            if (m < M && n < Nc) epilogue(ep, M, Nc, z, m, n, acc[i][j]);
        }
}

cudaError_t launch_gemm(int64_t M, int64_t Nc, int64_t K, const GemmOperand &A, const GemmOperand &Bm,
                        const GemmEpilogue &ep, int splits, cudaStream_t st) {
    if (M <= 0 || Nc <= 0) return cudaSuccess;
    if (splits < 1) splits = 1;
    int64_t kper = (K + splits - 1) / splits;
    kper = (kper + GB_K - 1) / GB_K * GB_K;
    dim3 grid(unsigned((Nc + GB_N - 1) / GB_N), unsigned((M + GB_M - 1) / GB_M), unsigned(splits));
    if (A.bf16 && Bm.bf16) k_gemm_simt<true, true><<<grid, 256, 0, st>>>(M, Nc, K, A, Bm, ep, kper);
    else if (A.bf16) k_gemm_simt<true, false><<<grid, 256, 0, st>>>(M, Nc, K, A, Bm, ep, kper);
    else if (Bm.bf16) k_gemm_simt<false, true><<<grid, 256, 0, st>>>(M, Nc, K, A, Bm, ep, kper);
    else k_gemm_simt<false, false><<<grid, 256, 0, st>>>(M, Nc, K, A, Bm, ep, kper);
    return cudaGetLastError();
}

}  // namespace adj
