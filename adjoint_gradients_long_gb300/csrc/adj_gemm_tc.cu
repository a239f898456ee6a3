// adj_gemm_tc.cu -- tcgen05 tensor-core GEMM with fused operand prologues and
// epilogues: C[M,Nc] = A[M,K] B[K,Nc], bf16 operands in shared memory, fp32
// accumulator in tensor memory.
//
// Two precisions:
//   BF16   operands rounded to bf16 (bf16 storage is used as is): one MMA per k-slice.
//   SPLIT3 fp32-accurate: every fp32 operand x is split into hi = bf16(x) and
//          lo = bf16(x - hi); the product uses hi*hi + hi*lo + lo*hi (the lo*lo
//          term is below 2^-16 of the product), three MMAs into one accumulator.
//
// CTA: 9 warps.  Warps 0-7 stage operand tiles (any stride, fp32 or bf16, optional
// elementwise product) into shared memory in the 128-byte-swizzled K-major layout,
// then run the epilogue.  Warp 8 owns the tensor memory and one of its lanes issues
// tcgen05.mma.  Stages are handed over with mbarriers: producers arrive on full[s];
// tcgen05.commit arrives on empty[s] when the MMAs reading stage s are done, and on
// `accum` after the last k-block.  Every wait is bounded by a wall-clock limit.
//
// Tile: BM = 128 rows (TMEM lanes), BN <= 256 columns (TMEM columns), BK = 64
// (one 128-byte swizzle row of bf16).  Shared-memory element (r, k) of a tile lives
// at byte r*128 + ((k/8) ^ (r%8))*16 + (k%8)*2 (8-row atoms of 1024 bytes).
#include "adj_internal.cuh"
#include "adj_epilogue.cuh"

namespace adj {

constexpr int TC_BM = 128, TC_BK = 64;
constexpr int TC_PROD_WARPS = 8, TC_PROD = TC_PROD_WARPS * 32, TC_THREADS = TC_PROD + 32;
constexpr unsigned long long TC_WAIT_NS = 2000000000ull;   // 2 s per wait

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false if the CTA aborted or the wait gave up (then records the timeout).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort, unsigned *status) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*abort) return false;
            const uint64_t t = gtimer();
            if (t0 == 0) t0 = t;
            else if (t - t0 > TC_WAIT_NS) {
                *abort = 1;
                record_timeout(status);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);          // start address
    d |= uint64_t(1) << 16;                          // leading byte offset (unused for this layout)
    d |= uint64_t(1024 >> 4) << 32;                  // stride byte offset: next 8-row atom
    d |= uint64_t(1) << 46;                          // descriptor version
    d |= uint64_t(2) << 61;                          // swizzle: 128 bytes
    return d;
}
// Instruction descriptor: kind::f16, bf16 x bf16 -> fp32, both operands K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(TC_BM >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- operand staging
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Write 8 consecutive-k values of row r (k chunk kc) as bf16 hi (and lo) into a tile.
template <bool SPLIT>
__device__ __forceinline__ void put8(uint8_t *hi, uint8_t *lo, int r, int kc, const float (&v)[8]) {
    const uint32_t off = uint32_t(r) * 128u + (uint32_t(kc ^ (r & 7)) << 4);
    uint4 h;
    h.x = pack_bf16(v[0], v[1]);
    h.y = pack_bf16(v[2], v[3]);
    h.z = pack_bf16(v[4], v[5]);
    h.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4 *>(hi + off) = h;
    if (SPLIT) {
        uint4 l;
        l.x = pack_bf16(v[0] - bf16_round(v[0]), v[1] - bf16_round(v[1]));
        l.y = pack_bf16(v[2] - bf16_round(v[2]), v[3] - bf16_round(v[3]));
        l.z = pack_bf16(v[4] - bf16_round(v[4]), v[5] - bf16_round(v[5]));
        l.w = pack_bf16(v[6] - bf16_round(v[6]), v[7] - bf16_round(v[7]));
        *reinterpret_cast<uint4 *>(lo + off) = l;
    }
}

template <bool BF>
__device__ __forceinline__ void ld8_contig(const void *p, int64_t i, float (&v)[8]) {
    if (BF) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + i));
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            v[2 * j] = f.x;
            v[2 * j + 1] = f.y;
        }
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}
template <bool BF>
__device__ __forceinline__ float ld1(const void *p, int64_t i) {
    if (BF) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    return __ldg(static_cast<const float *>(p) + i);
}

// Operand element addressing: A (IS_A) is split along k, B along its row index
// (its rows are output columns).  Returns the array and the element index.
template <bool IS_A>
__device__ __forceinline__ const void *op_at(const GemmOperand &O, int64_t row, int64_t k, int64_t &idx) {
    int blk;
    if (IS_A) {
        blk = int(k / O.blk);
        idx = row * O.s_row + (k - int64_t(blk) * O.blk) * O.s_k;
    } else {
        blk = int(row / O.blk);
        idx = (row - int64_t(blk) * O.blk) * O.s_row + k * O.s_k;
    }
    return O.p[blk];
}

// Stage rows [row0, row0+R) x k [k0, k0+64) of an operand into a swizzled tile.
// k-contiguous sources: a work item is 8 consecutive k of one row (two float4 or one
// 16-byte bf16 vector).  Row-contiguous sources (the token-major operands of the
// parameter reductions): a work item is a 4-row (fp32) or 8-row (bf16) by 8-k block,
// loaded as 8 row vectors and transposed in registers.  Loads of a thread's items are
// issued before any is converted, so several vectors are in flight per thread.
template <bool BF, bool SPLIT, bool IS_A>
__device__ __forceinline__ void stage_tile(const GemmOperand &O, int64_t row0, int64_t rows, int R, int64_t k0,
                                           int64_t kend, uint8_t *hi, uint8_t *lo, int tid) {
    constexpr int BATCH = 2;
    if (O.s_k == 1) {
        const int items = R * 8;
        for (int base_it = tid; base_it < items; base_it += TC_PROD * BATCH) {
            float v[BATCH][8];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int it = base_it + b * TC_PROD;
                const int r = it >> 3, kc = it & 7;
                const int64_t row = row0 + r, k = k0 + kc * 8;
                if (it < items && row < rows && k < kend) {
                    int64_t i;
                    const void *p = op_at<IS_A>(O, row, k, i);
                    if (k + 8 <= kend) {
                        ld8_contig<BF>(p, i, v[b]);
                        if (IS_A && O.mul) {
                            float m[8];
                            ld8_contig<false>(O.mul, i, m);
#pragma unroll
                            for (int j = 0; j < 8; ++j) v[b][j] *= m[j];
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            v[b][j] = (k + j < kend) ? ld1<BF>(p, i + j) : 0.f;
                            if (IS_A && O.mul && k + j < kend) v[b][j] *= __ldg(O.mul + i + j);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[b][j] = 0.f;
                }
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int it = base_it + b * TC_PROD;
                if (it < items) put8<SPLIT>(hi, lo, it >> 3, it & 7, v[b]);
            }
        }
        return;
    }
    // row-contiguous source: RB rows x 8 k per item
    constexpr int RB = BF ? 8 : 4;
    const int groups = R / RB, items = groups * 8;
    for (int it = tid; it < items; it += TC_PROD) {
        const int g = it % groups, kc = it / groups;
        const int r0 = g * RB;
        const int64_t row = row0 + r0, k = k0 + kc * 8;
        float v[RB][8];   // v[row][k]
        const bool full = row + RB <= rows && k + 8 <= kend;
        if (full) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int64_t i;
                const void *p = op_at<IS_A>(O, row, k + j, i);
                if (BF) {
                    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + i));
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
                    for (int q = 0; q < RB / 2; ++q) {
                        const float2 f = __bfloat1622float2(b2[q]);
                        v[2 * q][j] = f.x;
                        v[2 * q + 1][j] = f.y;
                    }
                } else {
                    const float4 f = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
                    v[0][j] = f.x; v[1 % RB][j] = f.y; v[2 % RB][j] = f.z; v[3 % RB][j] = f.w;
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < RB; ++q)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float x = 0.f;
                    if (row + q < rows && k + j < kend) {
                        int64_t i;
                        const void *p = op_at<IS_A>(O, row + q, k + j, i);
                        x = ld1<BF>(p, i);
                    }
                    v[q][j] = x;
                }
        }
#pragma unroll
        for (int q = 0; q < RB; ++q) put8<SPLIT>(hi, lo, r0 + q, kc, v[q]);
    }
}

// ---------------------------------------------------------------- the kernel
struct TcArgs {
    int64_t M, Nc, K, kper;
    int BN, stages;
    GemmOperand A, Bm;
    GemmEpilogue ep;
    unsigned *status;
};

template <bool ABF, bool BBF, bool SPLIT>
__global__ void __launch_bounds__(TC_THREADS, 1) k_gemm_tc(const TcArgs args) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned stage buffers, then barriers
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int BN = args.BN, S = args.stages;
    const uint32_t a_bytes = TC_BM * 128, b_bytes = uint32_t(BN) * 128;
    const uint32_t stage_bytes = (a_bytes + b_bytes) * (SPLIT ? 2 : 1);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + size_t(S) * stage_bytes);
    uint64_t *full = bars, *empty = bars + S, *accum = bars + 2 * S;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(bars + 2 * S + 1) + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t m0 = int64_t(blockIdx.y) * TC_BM, n0 = int64_t(blockIdx.x) * BN;
    const int z = blockIdx.z;
    const int64_t kbeg = int64_t(z) * args.kper;
    const int64_t kend = kbeg + args.kper < args.K ? kbeg + args.kper : args.K;
    const int nkb = kend > kbeg ? int((kend - kbeg + TC_BK - 1) / TC_BK) : 0;
    uint32_t ncols = 32;
    while (ncols < uint32_t(BN)) ncols <<= 1;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), TC_PROD);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accum), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == TC_PROD_WARPS) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(const_cast<uint32_t *>(tmem_slot))),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < TC_PROD_WARPS) {
        // ---------------- producers
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % S, r = kb / S;
            if (r > 0 && !mbar_wait(smem_u32(&empty[s]), (r - 1) & 1, abort, args.status)) break;
            uint8_t *st = base + size_t(s) * stage_bytes;
            uint8_t *a_hi = st, *b_hi = st + a_bytes;
            uint8_t *a_lo = SPLIT ? st + a_bytes + b_bytes : nullptr;
            uint8_t *b_lo = SPLIT ? a_lo + a_bytes : nullptr;
            const int64_t k0 = kbeg + int64_t(kb) * TC_BK;
            stage_tile<ABF, SPLIT, true>(args.A, m0, args.M, TC_BM, k0, kend, a_hi, a_lo, tid);
            stage_tile<BBF, SPLIT, false>(args.Bm, n0, args.Nc, BN, k0, kend, b_hi, b_lo, tid);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&full[s]));
        }
        // ---------------- epilogue: warp w reads TMEM lanes 32*(w%4).., column chunks (w/4), (w/4)+2, ...
        // Each 32 x 32 chunk goes through shared memory (the drained stage buffers) so that
        // the stores of a warp cover one output row segment of 32 consecutive columns.
        const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(accum), 0, abort, args.status));
        tc_fence_after();
        float *sbuf = reinterpret_cast<float *>(base) + warp * (32 * 33);
        const int q = warp & 3;
        for (int c = (warp >> 2) * 32; c < BN; c += 64) {
            float v[32];
            if (ok && nkb > 0) {
                tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(c), v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) sbuf[lane * 33 + j] = v[j];
            __syncwarp();
            const int n = int(n0) + c + lane;
            if (n < args.Nc) {
                for (int i = 0; i < 32; ++i) {
                    const int64_t m = m0 + q * 32 + i;
                    if (m < args.M) epilogue(args.ep, args.M, args.Nc, z, m, n, sbuf[i * 33 + lane]);
                }
            }
            __syncwarp();
        }
    } else if (lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = idesc_bf16(BN);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % S, r = kb / S;
            if (!mbar_wait(smem_u32(&full[s]), r & 1, abort, args.status)) break;
            tc_fence_after();
            const uint32_t st = smem_u32(base + size_t(s) * stage_bytes);
            const uint32_t a_hi = st, b_hi = st + a_bytes;
            const uint32_t a_lo = st + a_bytes + b_bytes, b_lo = a_lo + a_bytes;
#pragma unroll
            for (int ks = 0; ks < TC_BK / 16; ++ks) {
                const uint32_t koff = uint32_t(ks) * 32u;
                const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
                mma_bf16(tmem, sw128_desc(a_hi + koff), sw128_desc(b_hi + koff), idesc, acc);
                if (SPLIT) {
                    mma_bf16(tmem, sw128_desc(a_hi + koff), sw128_desc(b_lo + koff), idesc, 1u);
                    mma_bf16(tmem, sw128_desc(a_lo + koff), sw128_desc(b_hi + koff), idesc, 1u);
                }
            }
            mma_commit(smem_u32(&empty[s]));
        }
        mma_commit(smem_u32(accum));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == TC_PROD_WARPS) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

// ---------------------------------------------------------------- launcher
static size_t tc_smem_bytes(int BN, int stages, bool split) {
    const size_t stage = size_t(TC_BM * 128 + BN * 128) * (split ? 2 : 1);
    return 1024 + stage * stages + (2 * stages + 2) * 8 + 64;
}

template <bool ABF, bool BBF, bool SPLIT>
static cudaError_t launch_tc_t(const TcArgs &a, dim3 grid, size_t smem, cudaStream_t st) {
    auto kern = k_gemm_tc<ABF, BBF, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, TC_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tc(int64_t M, int64_t Nc, int64_t K, const GemmOperand &A, const GemmOperand &Bm,
                           const GemmEpilogue &ep, int splits, bool split3, unsigned *status, cudaStream_t st) {
    if (M <= 0 || Nc <= 0) return cudaSuccess;
    if (splits < 1) splits = 1;
    TcArgs a;
    a.M = M; a.Nc = Nc; a.K = K;
    int64_t kper = (K + splits - 1) / splits;
    a.kper = (kper + TC_BK - 1) / TC_BK * TC_BK;
    const int nkb = int((a.kper + TC_BK - 1) / TC_BK);
    // Short reductions (a few k-blocks per tile) with many tiles: 128-column tiles, so two
    // CTAs fit per SM and one's loads overlap the other's epilogue.
    const int64_t tiles256 = ((Nc + 255) / 256) * ((M + TC_BM - 1) / TC_BM) * splits;
    int BN = int(Nc < 256 ? (Nc + 31) / 32 * 32 : 256);
    if (BN > 128 && nkb <= 4 && tiles256 >= 2 * 152) BN = 128;
    a.BN = BN;
    const int max_stages = split3 ? 2 : 4;
    a.stages = nkb < 1 ? 1 : (nkb < max_stages ? nkb : max_stages);
    a.A = A; a.Bm = Bm; a.ep = ep; a.status = status;
    const size_t smem = tc_smem_bytes(BN, a.stages, split3);
    dim3 grid(unsigned((Nc + BN - 1) / BN), unsigned((M + TC_BM - 1) / TC_BM), unsigned(splits));
    if (split3) {
        if (A.bf16 && Bm.bf16) return launch_tc_t<true, true, true>(a, grid, smem, st);
        if (A.bf16) return launch_tc_t<true, false, true>(a, grid, smem, st);
        if (Bm.bf16) return launch_tc_t<false, true, true>(a, grid, smem, st);
        return launch_tc_t<false, false, true>(a, grid, smem, st);
    }
    if (A.bf16 && Bm.bf16) return launch_tc_t<true, true, false>(a, grid, smem, st);
    if (A.bf16) return launch_tc_t<true, false, false>(a, grid, smem, st);
    if (Bm.bf16) return launch_tc_t<false, true, false>(a, grid, smem, st);
    return launch_tc_t<false, false, false>(a, grid, smem, st);
}

}  // namespace adj
