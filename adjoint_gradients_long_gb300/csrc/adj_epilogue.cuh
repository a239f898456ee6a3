// adj_epilogue.cuh -- the fused GEMM epilogues shared by the GEMM kernels:
//   ProjIn   columns [0,N) -> a = sigmoid(acc + b_a), [N,2N) -> u, [2N,3N) -> c
//   Store    out0[m,n] = acc (+ bf16 copy)
//   StoreAdd out0[m,n] = acc + add[m,n] (+ bf16 copy)
//   Partial  out0[z][m][n] = acc (split-K partial z)
#pragma once
#include "adj_internal.cuh"

namespace adj {

__device__ __forceinline__ void epilogue(const GemmEpilogue &ep, int64_t M, int64_t Nc, int z, int64_t m,
                                         int64_t n, float acc) {
    switch (ep.kind) {
    case Epi::ProjIn: {
        const int nn = int(n), blk = nn / ep.N;
        const int j = nn - blk * ep.N;
        if (blk == 0) ep.out0[m * ep.N + j] = 1.f / (1.f + expf(-(acc + ep.bias[j])));
        else if (blk == 1) ep.out1[m * ep.N + j] = acc;
        else ep.out2[m * ep.N + j] = acc;
        break;
    }
    case Epi::Store:
    case Epi::StoreAdd: {
        float v = acc;
        if (ep.kind == Epi::StoreAdd)
            v += ep.add_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(ep.add)[m * ep.ld + n])
                             : static_cast<const float *>(ep.add)[m * ep.ld + n];
        ep.out0[m * ep.ld + n] = v;
        if (ep.out_x) static_cast<__nv_bfloat16 *>(ep.out_x)[m * ep.ld + n] = __float2bfloat16_rn(v);
        break;
    }
    case Epi::Partial:
        ep.out0[(int64_t(z) * M + m) * Nc + n] = acc;
        break;
    }
}


}  // namespace adj
