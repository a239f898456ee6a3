// adj_misc.cu -- reductions of the adjoint-sharding path: the loss and its cotangent,
// the column sum db_a = sum_t D_a, and the deterministic split-K reduction of the
// parameter-gradient partials.  All are coalesced, 128-bit where the layout allows.
#include "adj_internal.cuh"

namespace adj {

// ---------------------------------------------------------------- loss
// L = sum 1/2 (y - target)^2, gy = y - target; one fp64 partial per block, then one
// block sums the partials in a fixed order (deterministic).
__global__ void __launch_bounds__(256) k_loss(const float *__restrict__ y, const float *__restrict__ tg,
                                              float *__restrict__ gy, int64_t count, double *__restrict__ part) {
    __shared__ double red[256];
    double s = 0.0;
    const int64_t n4 = count / 4;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4 r = ld_stream4(y + 4 * i) - ld_stream4(tg + 4 * i);
        if (gy) st_stream4(gy + 4 * i, r);
        s += 0.5 * (double(r.x) * r.x + double(r.y) * r.y + double(r.z) * r.z + double(r.w) * r.w);
    }
    for (int64_t i = 4 * n4 + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float r = y[i] - tg[i];
        if (gy) gy[i] = r;
        s += 0.5 * double(r) * r;
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) part[blockIdx.x] = red[0];
}

__global__ void k_sum_partials(const double *__restrict__ part, int n, double *__restrict__ out) {
    __shared__ double red[256];
    double s = 0.0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s += part[i];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = red[0];
}

cudaError_t launch_loss(const float *y, const float *target, float *gy, int64_t count, double *part, int nblk,
                        double *loss, cudaStream_t st) {
    k_loss<<<nblk, 256, 0, st>>>(y, target, gy, count, part);
    if (loss) k_sum_partials<<<1, 256, 0, st>>>(part, nblk, loss);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- column sums
// part[blk][n] = sum over the block's rows of D[row][n]; out[n] (+)= sum_blk part[blk][n].
template <bool BF>
__global__ void __launch_bounds__(256) k_colsum(const void *__restrict__ D, int64_t rows, int N,
                                                int64_t rows_per_blk, float *__restrict__ part) {
    const int64_t r0 = blockIdx.x * rows_per_blk;
    const int64_t r1 = r0 + rows_per_blk < rows ? r0 + rows_per_blk : rows;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        float s = 0.f;
        for (int64_t r = r0; r < r1; ++r) {
            if (BF) s += __bfloat162float(static_cast<const __nv_bfloat16 *>(D)[r * N + n]);
            else s += static_cast<const float *>(D)[r * N + n];
        }
        part[int64_t(blockIdx.x) * N + n] = s;
    }
}

__global__ void k_colsum_final(const float *__restrict__ part, int nblk, int N, float *__restrict__ out,
                               int accumulate) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    float s = 0.f;
    for (int b = 0; b < nblk; ++b) s += part[int64_t(b) * N + n];
    out[n] = accumulate ? out[n] + s : s;
}

cudaError_t launch_colsum(const void *D, bool bf16, int64_t rows, int N, float *part, int nblk, float *out,
                          int accumulate, cudaStream_t st) {
    const int64_t rpb = (rows + nblk - 1) / nblk;
    if (bf16) k_colsum<true><<<nblk, 256, 0, st>>>(D, rows, N, rpb, part);
    else k_colsum<false><<<nblk, 256, 0, st>>>(D, rows, N, rpb, part);
    k_colsum_final<<<(N + 255) / 256, 256, 0, st>>>(part, nblk, N, out, accumulate);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- split-K reduction
__global__ void __launch_bounds__(256) k_splitk_reduce(const float *__restrict__ part, int splits, int64_t count,
                                                       float *__restrict__ out, int accumulate) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count; i += int64_t(gridDim.x) * blockDim.x) {
        float s = accumulate ? out[i] : 0.f;
        for (int z = 0; z < splits; ++z) s += part[int64_t(z) * count + i];
        out[i] = s;
    }
}

cudaError_t launch_splitk_reduce(const float *part, int splits, int64_t count, float *out, int accumulate,
                                 cudaStream_t st) {
    int64_t blocks = (count + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_splitk_reduce<<<unsigned(blocks), 256, 0, st>>>(part, splits, count, out, accumulate);
    return cudaGetLastError();
}

}  // namespace adj
