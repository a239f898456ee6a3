// adj_misc.cu -- reductions of the adjoint-sharding path: the loss and its cotangent,
// the column sum db_a = sum_t D_a, and the deterministic split-K reduction of the
// parameter-gradient partials.  All are coalesced, 128-bit where the layout allows.
#include "adj_internal.cuh"

namespace adj {

// ---------------------------------------------------------------- loss
// L = sum 1/2 (y - target)^2, gy = y - target.  Each thread sums its elements in fp32
// (a few dozen terms), the block combines the thread sums in fp64 and writes one
// partial; the block that finishes last (a wrapping ticket in the workspace header,
// back at zero after every launch) sums the partials in a fixed order, so the result
// does not depend on block order.  FP64 arithmetic is kept out of the per-element loop:
// GB300's fp64 rate is a small fraction of its fp32 rate.
__global__ void __launch_bounds__(256) k_loss(const float *__restrict__ y, const float *__restrict__ tg,
                                              float *__restrict__ gy, __nv_bfloat16 *__restrict__ gyx, int64_t count,
                                              double *__restrict__ part, unsigned *ticket, double *__restrict__ loss) {
    __shared__ double red[256];
    __shared__ bool last;
    float s = 0.f;
    const int64_t n4 = count / 4, stride = int64_t(gridDim.x) * blockDim.x;
    int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    // four vectors of each input in flight per thread
    for (; i + 3 * stride < n4; i += 4 * stride) {
        float4 a[4], b[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            a[u] = ld_stream4(y + 4 * (i + u * stride));
            b[u] = ld_stream4(tg + 4 * (i + u * stride));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float4 r = a[u] - b[u];
            if (gy) st4(gy + 4 * (i + u * stride), r);   // kept in L2: the cotangent projection reads gy next
            if (gyx) st4(gyx + 4 * (i + u * stride), r);
            s += 0.5f * (r.x * r.x + r.y * r.y + r.z * r.z + r.w * r.w);
        }
    }
    for (; i < n4; i += stride) {
        const float4 r = ld_stream4(y + 4 * i) - ld_stream4(tg + 4 * i);
        if (gy) st4(gy + 4 * i, r);
        if (gyx) st4(gyx + 4 * i, r);
        s += 0.5f * (r.x * r.x + r.y * r.y + r.z * r.z + r.w * r.w);
    }
    for (int64_t i = 4 * n4 + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float r = y[i] - tg[i];
        if (gy) gy[i] = r;
        if (gyx) gyx[i] = __float2bfloat16_rn(r);
        s += 0.5f * r * r;
    }
    red[threadIdx.x] = double(s);
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (!loss) return;
    if (threadIdx.x == 0) {
        part[blockIdx.x] = red[0];
        __threadfence();
        last = atomicInc(ticket, gridDim.x - 1) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    double t = 0.0;
    for (int i = threadIdx.x; i < int(gridDim.x); i += blockDim.x) t += __ldcg(&part[i]);
    red[threadIdx.x] = t;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) *loss = red[0];
}

cudaError_t launch_loss(const float *y, const float *target, float *gy, __nv_bfloat16 *gyx, int64_t count, double *part,
                        int nblk, unsigned *ticket, double *loss, cudaStream_t st) {
    k_loss<<<nblk, 256, 0, st>>>(y, target, gy, gyx, count, part, ticket, loss);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- column sums
// part[blk][n] = sum over the block's rows of D[row][n]; the blocks own contiguous row
// ranges and their partials are summed by k_reduce_partials.  A block is 256 threads =
// (N/4 column groups of 4) x (256/(N/4) row lanes); each thread reads 4 columns (one 8- or
// 16-byte vector) of every row-lane-th row, eight rows in flight, and the row lanes are
// combined in shared memory in a fixed order.
template <bool BF>
__device__ __forceinline__ float4 ld_row4(const void *D, int64_t i) {
    if (BF) {
        const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(D) + i));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    return ld_stream4(static_cast<const float *>(D) + i);
}

template <bool BF>
__global__ void __launch_bounds__(256) k_colsum(const void *__restrict__ D, int64_t rows, int N,
                                                int64_t rows_per_blk, float *__restrict__ part) {
    __shared__ float4 red[256];
    const int groups = N / 4 < 256 ? N / 4 : 256;   // column groups handled at once
    const int lanes = 256 / groups;                  // row lanes
    const int gq = threadIdx.x % groups, rl = threadIdx.x / groups;
    const int64_t r0 = blockIdx.x * rows_per_blk;
    const int64_t r1 = r0 + rows_per_blk < rows ? r0 + rows_per_blk : rows;
    for (int c0 = 0; c0 < N; c0 += groups * 4) {
        const int col = c0 + gq * 4;
        float4 acc = f4(0.f);
        if (rl < lanes && col < N) {
            int64_t r = r0 + rl;
            for (; r + 7 * lanes < r1; r += 8 * lanes) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = ld_row4<BF>(D, (r + u * lanes) * N + col);
                acc = acc + (((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7])));
            }
            for (; r < r1; r += lanes) acc = acc + ld_row4<BF>(D, r * N + col);
        }
        red[threadIdx.x] = acc;
        __syncthreads();
        if (threadIdx.x < groups && col < N) {
            float4 t = f4(0.f);
            for (int l = 0; l < lanes; ++l) t = t + red[l * groups + threadIdx.x];
            *reinterpret_cast<float4 *>(part + int64_t(blockIdx.x) * N + col) = t;
        }
        __syncthreads();
    }
}

cudaError_t launch_colsum(const void *D, bool bf16, int64_t rows, int N, float *part, int nblk, cudaStream_t st) {
    const int64_t rpb = (rows + nblk - 1) / nblk;
    if (bf16) k_colsum<true><<<nblk, 256, 0, st>>>(D, rows, N, rpb, part);
    else k_colsum<false><<<nblk, 256, 0, st>>>(D, rows, N, rpb, part);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- partial reductions
// out[i] (+)= sum_z part[z][i] for up to three independent arrays (the split-K partials of
// dW_in and dW_o, the column-sum partials of db_a) in one launch; each array owns a range
// of blocks.  Wide arrays with more than 32 partials: a block covers 32 consecutive float4
// outputs, warp w sums the partials z = w, w + 8, ... (eight loads in flight, every load a
// 512-byte row segment) and the eight warp sums are added in warp order.  Narrow arrays
// (the column sums) and wide arrays with at most 32 partials (the split-K products): an
// output float4 is owned by a group of G lanes (a power of two, at most 32, so that a lane
// loads at most eight partials at a time), or by a whole block when 32 lanes would need
// more; lane g sums z = g, g + G, ... and a butterfly of
// shuffles combines the group (then shared memory, in warp order, for a block).  The order of every addition
// is fixed, so the result does not depend on scheduling.
__global__ void __launch_bounds__(256) k_reduce_partials(RedArgs r) {
    // the array by explicit selection (an indexed parameter array would go to local memory)
    const int64_t bx = blockIdx.x;
    const bool s2 = r.nseg > 2 && bx >= r.seg[2].first, s1 = !s2 && r.nseg > 1 && bx >= r.seg[1].first;
    const float4 *part = reinterpret_cast<const float4 *>(s2 ? r.seg[2].part : s1 ? r.seg[1].part : r.seg[0].part);
    float4 *out = reinterpret_cast<float4 *>(s2 ? r.seg[2].out : s1 ? r.seg[1].out : r.seg[0].out);
    const int64_t n4 = s2 ? r.seg[2].n4 : s1 ? r.seg[1].n4 : r.seg[0].n4;
    const int64_t blk = bx - (s2 ? r.seg[2].first : s1 ? r.seg[1].first : r.seg[0].first);
    const int splits = s2 ? r.seg[2].splits : s1 ? r.seg[1].splits : r.seg[0].splits;
    const int G = s2 ? r.seg[2].group : s1 ? r.seg[1].group : r.seg[0].group;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float4 red[8][32];
    if (G == 0) {
        const int64_t q = blk * 32 + lane;
        float4 s = f4(0.f);
        if (q < n4) {
            for (int z0 = w; z0 < splits; z0 += 64) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int z = z0 + 8 * u;
                    v[u] = z < splits ? __ldcs(part + int64_t(z) * n4 + q) : f4(0.f);
                }
                s = s + (((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7])));
            }
        }
        red[w][lane] = s;
        __syncthreads();
        if (w == 0 && q < n4) {
            float4 t = red[0][lane];
#pragma unroll
            for (int k = 1; k < 8; ++k) t = t + red[k][lane];
            if (r.accumulate) t = out[q] + t;
            out[q] = t;
        }
        return;
    }
    if (G == 256) {
        // one block per output float4: thread t sums z = t, t + 256, ..., then a shuffle
        // butterfly in each warp and the eight warp sums in warp order
        const int64_t q = blk;
        const float4 *p = part + q;
        float4 s = f4(0.f);
        for (int z0 = threadIdx.x; z0 < splits; z0 += 8 * 256) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int z = z0 + u * 256;
                v[u] = z < splits ? __ldcs(p + int64_t(z) * n4) : f4(0.f);
            }
            s = s + (((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7])));
        }
        for (int o = 1; o < 32; o <<= 1) {
            s.x += __shfl_xor_sync(0xffffffffu, s.x, o);
            s.y += __shfl_xor_sync(0xffffffffu, s.y, o);
            s.z += __shfl_xor_sync(0xffffffffu, s.z, o);
            s.w += __shfl_xor_sync(0xffffffffu, s.w, o);
        }
        if (lane == 0) red[w][0] = s;
        __syncthreads();
        if (threadIdx.x == 0) {
            float4 t = red[0][0];
#pragma unroll
            for (int k = 1; k < 8; ++k) t = t + red[k][0];
            if (r.accumulate) t = out[q] + t;
            out[q] = t;
        }
        return;
    }
    const int64_t q = blk * (256 / G) + threadIdx.x / G;
    const int g = threadIdx.x % G;
    const bool live = q < n4;
    float4 s = f4(0.f);
    if (live) {
        const float4 *p = part + q;
        for (int z0 = g; z0 < splits; z0 += 8 * G) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int z = z0 + u * G;
                v[u] = z < splits ? __ldcs(p + int64_t(z) * n4) : f4(0.f);
            }
            s = s + (((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7])));
        }
    }
    for (int o = 1; o < G; o <<= 1) {
        s.x += __shfl_xor_sync(0xffffffffu, s.x, o);
        s.y += __shfl_xor_sync(0xffffffffu, s.y, o);
        s.z += __shfl_xor_sync(0xffffffffu, s.z, o);
        s.w += __shfl_xor_sync(0xffffffffu, s.w, o);
    }
    if (live && g == 0) {
        if (r.accumulate) s = out[q] + s;
        out[q] = s;
    }
}

cudaError_t launch_reduce_partials(const RedSeg *segs, int nseg, int accumulate, cudaStream_t st) {
    RedArgs r;
    memset(&r, 0, sizeof(r));
    if (nseg < 1 || nseg > 3) return cudaErrorInvalidValue;
    int64_t first = 0;
    for (int k = 0; k < nseg; ++k) {
        r.seg[k] = segs[k];
        int G = 0;                                   // 0: warps over the partials
        // narrow arrays, or few partials (a wide array's warps would mostly idle over them):
        // lane groups, or whole blocks
        if (segs[k].n4 < 4096 || segs[k].splits <= 32) {
            G = 1;
            while (G < 32 && (segs[k].splits + G - 1) / G > 8) G <<= 1;
            if ((segs[k].splits + G - 1) / G > 8) G = 256;
        }
        r.seg[k].group = G;
        r.seg[k].first = first;                      // first block of the array
        first += G == 0 ? (segs[k].n4 + 31) / 32 : G == 256 ? segs[k].n4 : (segs[k].n4 * G + 255) / 256;
    }
    r.nseg = nseg;
    r.accumulate = accumulate;
    if (first < 1) return cudaSuccess;
    k_reduce_partials<<<unsigned(first), 256, 0, st>>>(r);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- bf16 hi/lo split of an operand
__global__ void __launch_bounds__(256) k_split_bf16(const float *__restrict__ w, int64_t n,
                                                    __nv_bfloat16 *__restrict__ hi, __nv_bfloat16 *__restrict__ lo) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const float x = w[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        hi[i] = h;
        lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
    }
}

__global__ void __launch_bounds__(256) k_prep_win(const void *__restrict__ w, bool w_bf16, int P, int N,
                                                  __nv_bfloat16 *__restrict__ hi, __nv_bfloat16 *__restrict__ lo,
                                                  const float *__restrict__ wo, int64_t n_wo,
                                                  __nv_bfloat16 *__restrict__ wo_hi, __nv_bfloat16 *__restrict__ wo_lo) {
    const int64_t n3 = 3 * int64_t(N), total = int64_t(P) * n3;
    // the forward's other weight in the same launch: W_o split into bf16 hi and lo
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_wo; i += int64_t(gridDim.x) * blockDim.x) {
        const float x = wo[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        wo_hi[i] = h;
        wo_lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
    }
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t p = i / n3;
        const int c = int(i - p * n3), j = c >> 5;
        const int64_t src = p * n3 + int64_t(j % 3) * N + (j / 3) * 32 + (c & 31);
        if (w_bf16) {
            hi[i] = static_cast<const __nv_bfloat16 *>(w)[src];
        } else {
            const float x = static_cast<const float *>(w)[src];
            const __nv_bfloat16 h = __float2bfloat16_rn(x);
            hi[i] = h;
            lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
        }
    }
}

cudaError_t launch_prep_win(const void *w, bool w_bf16, int P, int N, __nv_bfloat16 *hi, __nv_bfloat16 *lo,
                            cudaStream_t st, const float *wo, __nv_bfloat16 *wo_hi, __nv_bfloat16 *wo_lo) {
    int64_t blocks = (int64_t(P) * 3 * N + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) return cudaSuccess;
    const int64_t n_wo = wo ? int64_t(N) * P : 0;
    k_prep_win<<<unsigned(blocks), 256, 0, st>>>(w, w_bf16, P, N, hi, lo, wo, n_wo, wo_hi, wo_lo);
    return cudaGetLastError();
}

cudaError_t launch_split_bf16(const float *w, int64_t n, __nv_bfloat16 *hi, __nv_bfloat16 *lo, cudaStream_t st) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) return cudaSuccess;
    k_split_bf16<<<unsigned(blocks), 256, 0, st>>>(w, n, hi, lo);
    return cudaGetLastError();
}

}  // namespace adj

namespace adj {

// ---------------------------------------------------------------- normalised layer inputs
// xhat = y / r, r = sqrt(mean_p y_p^2 + eps), per token row; one warp per row, the row
// read as float4 (P is a multiple of 8).
template <bool XBF>
__global__ void __launch_bounds__(256) k_rms_norm(const float *__restrict__ y, void *__restrict__ xhat,
                                                  float *__restrict__ r, int64_t rows, int P, float eps) {
    const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *yr = y + row * P;
    float ss = 0.f;
    for (int p = lane * 4; p < P; p += 128) {
        const float4 v = ld_keep4(yr + p);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rr = sqrtf(ss / float(P) + eps), inv = 1.f / rr;
    for (int p = lane * 4; p < P; p += 128) {
        const float4 v = ld_keep4(yr + p) * f4(inv);
        if (XBF) st4(static_cast<__nv_bfloat16 *>(xhat) + row * P + p, v);
        else st4(static_cast<float *>(xhat) + row * P + p, v);
    }
    if (lane == 0) r[row] = rr;
}

// gy_prev = gy + (dx - xhat mean_p(xhat dx)) / r with xhat = y / r recomputed in fp32.
// gy_prev may alias dx or gy (each element is read before it is written, by one lane).
__global__ void __launch_bounds__(256) k_rms_norm_bwd(const float *__restrict__ y, const float *__restrict__ r,
                                                      const float *dx, const float *gy, float *gy_prev,
                                                      int64_t rows, int P) {
    const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float inv = 1.f / r[row];
    const float *yr = y + row * P;
    const float *dr = dx + row * P;
    float s = 0.f;
    for (int p = lane * 4; p < P; p += 128) {
        const float4 xv = ld_keep4(yr + p) * f4(inv), dv = *reinterpret_cast<const float4 *>(dr + p);
        s += xv.x * dv.x + xv.y * dv.y + xv.z * dv.z + xv.w * dv.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float4 m = f4(s / float(P));
    for (int p = lane * 4; p < P; p += 128) {
        const float4 xv = ld_keep4(yr + p) * f4(inv);
        const float4 dv = *reinterpret_cast<const float4 *>(dr + p);
        const float4 gv = *reinterpret_cast<const float4 *>(gy + row * P + p);
        *reinterpret_cast<float4 *>(gy_prev + row * P + p) = gv + (dv - xv * m) * f4(inv);
    }
}

// The same with the row held in registers (NV float4 a lane, P = 128 NV): every byte of y
// is read from HBM once and all of a row's loads are in flight together.
template <bool XBF, int NV>
__global__ void __launch_bounds__(256) k_rms_norm_reg(const float *__restrict__ y, void *__restrict__ xhat,
                                                      float *__restrict__ r, int64_t rows, float eps) {
    constexpr int P = 128 * NV;
    const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *yr = y + row * P;
    float4 v[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = ld_stream4(yr + lane * 4 + j * 128);
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rr = sqrtf(ss / float(P) + eps), inv = 1.f / rr;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const float4 w = v[j] * f4(inv);
        if (XBF) st4(static_cast<__nv_bfloat16 *>(xhat) + row * P + lane * 4 + j * 128, w);
        else st4(static_cast<float *>(xhat) + row * P + lane * 4 + j * 128, w);
    }
    if (lane == 0) r[row] = rr;
}

cudaError_t launch_rms_norm(const float *y, void *xhat, bool xbf, float *r, int64_t rows, int P, float eps,
                            cudaStream_t st) {
    const unsigned grid = unsigned((rows + 7) / 8);
#define ADJ_RMS_REG(NV)                                                                    \
    do {                                                                                   \
        if (xbf) k_rms_norm_reg<true, NV><<<grid, 256, 0, st>>>(y, xhat, r, rows, eps);    \
        else k_rms_norm_reg<false, NV><<<grid, 256, 0, st>>>(y, xhat, r, rows, eps);       \
        return cudaGetLastError();                                                         \
    } while (0)
    switch (P) {
    case 256: ADJ_RMS_REG(2);
    case 512: ADJ_RMS_REG(4);
    case 1024: ADJ_RMS_REG(8);
    case 2048: ADJ_RMS_REG(16);
    default: break;
    }
#undef ADJ_RMS_REG
    if (xbf) k_rms_norm<true><<<grid, 256, 0, st>>>(y, xhat, r, rows, P, eps);
    else k_rms_norm<false><<<grid, 256, 0, st>>>(y, xhat, r, rows, P, eps);
    return cudaGetLastError();
}

cudaError_t launch_rms_norm_bwd(const float *y, const float *r, const float *dx, const float *gy, float *gy_prev,
                                int64_t rows, int P, cudaStream_t st) {
    k_rms_norm_bwd<<<unsigned((rows + 7) / 8), 256, 0, st>>>(y, r, dx, gy, gy_prev, rows, P);
    return cudaGetLastError();
}

}  // namespace adj
