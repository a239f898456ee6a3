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
#include "adj_ptx.cuh"

namespace adj {

#ifndef ADJ_TC_PROD_WARPS
#define ADJ_TC_PROD_WARPS 8
#endif
constexpr int TC_BM = 128, TC_BK = 64;
constexpr int TC_PROD_WARPS = ADJ_TC_PROD_WARPS, TC_PROD = TC_PROD_WARPS * 32;

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
    if (O.blk >= (int64_t(1) << 30)) {          // one array
        idx = row * O.s_row + k * O.s_k;
        return O.p[0];
    }
    const int bsz = int(O.blk);
    if (IS_A) {
        const int kk = int(k), blk = kk / bsz;
        idx = row * O.s_row + int64_t(kk - blk * bsz) * O.s_k;
        return O.p[blk];
    }
    const int rr = int(row), blk = rr / bsz;
    idx = int64_t(rr - blk * bsz) * O.s_row + k * O.s_k;
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
// Persistent and warp-specialised.  A CTA walks the output tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... (t -> m tile t / n_tiles, n tile t % n_tiles, with the
// split index outermost); gridDim.x is a multiple of n_tiles, so a CTA keeps one n tile.
// When the whole K extent of that n tile's B operand fits (B_RES), B is staged once and
// stays resident; otherwise B streams with A.
//   warps 0-7   epilogue: warp w reads TMEM lanes 32*(w%4).. for column half w/4, through
//               shared memory, 16-byte coalesced stores
//   warps 8-15  producers: stage A (and B) k-blocks into a ring of S stages
//   warp 16     TMEM owner; lane 0 issues tcgen05.mma into one of two accumulators
// Barriers: full[s]/empty[s] hand stages producer -> MMA -> producer; accf[b]/acce[b]
// hand accumulator b MMA -> epilogue -> MMA; bres marks the resident B tile ready.
constexpr int TC_EPI_WARPS = 8, TC_THREADS_P = (TC_EPI_WARPS + TC_PROD_WARPS + 1) * 32;
constexpr int TC_MMA_WARP = TC_EPI_WARPS + TC_PROD_WARPS;
constexpr uint32_t TC_EPI_SMEM = TC_EPI_WARPS * 32 * 32 * 4;

struct TcArgs {
    int64_t M, Nc, K, kper;
    int BN, stages, n_tiles, m_tiles, splits;
    bool b_res;
    GemmOperand A, Bm;
    GemmEpilogue ep;
    unsigned *status;
};

struct TcLayout {
    uint32_t a_bytes, b_bytes, stage_bytes, bres_bytes;
};
__host__ __device__ inline TcLayout tc_layout(int BN, int64_t K, bool b_res, bool split) {
    TcLayout L;
    const uint32_t f = split ? 2u : 1u;
    L.a_bytes = TC_BM * 128u;
    L.b_bytes = uint32_t(BN) * 128u;
    L.stage_bytes = (L.a_bytes + (b_res ? 0u : L.b_bytes)) * f;
    const uint32_t kb = uint32_t((K + TC_BK - 1) / TC_BK);
    L.bres_bytes = b_res ? L.b_bytes * kb * f : 0u;
    return L;
}

// Epilogue of one 32-row x 32-column chunk held in shared memory: row r, column quad q
// (columns 4q..4q+3) at float offset r*32 + 4*(q ^ (r%8)) (conflict-free both ways).
// Lane l owns quad l%8 of rows l/8, l/8+4, ...: every store is a 16-byte vector and a
// warp writes four full 128-byte row segments per instruction.
__device__ __forceinline__ int epi_at(int r, int q) { return r * 32 + ((q ^ (r & 7)) << 2); }

__device__ __forceinline__ float sigmoidf_fast(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

__device__ __forceinline__ void epi_chunk(const TcArgs &args, const float *sb, int64_t m0r, int n0c, int z, int lane) {
    const GemmEpilogue &ep = args.ep;
    const int64_t M = args.M;
    const int cq = (lane & 7) * 4, n = n0c + cq;
    if (n >= args.Nc) return;                    // Nc is a multiple of 8: a column quad is all in or all out
    const int rows = M - m0r < 32 ? int(M - m0r) : 32;
    switch (ep.kind) {
    case Epi::ProjIn: {
        const int blk = n / ep.N, j = n - blk * ep.N;
        float *out = (blk == 0 ? ep.out0 : blk == 1 ? ep.out1 : ep.out2) + m0r * ep.N + j;
        const float4 bias = blk == 0 ? *reinterpret_cast<const float4 *>(ep.bias + j) : f4(0.f);
        for (int i = lane >> 3; i < rows; i += 4) {
            float4 v = *reinterpret_cast<const float4 *>(sb + epi_at(i, lane & 7));
            if (blk == 0) {
                v.x = sigmoidf_fast(v.x + bias.x);
                v.y = sigmoidf_fast(v.y + bias.y);
                v.z = sigmoidf_fast(v.z + bias.z);
                v.w = sigmoidf_fast(v.w + bias.w);
            }
            st_stream4(out + int64_t(i) * ep.N, v);
        }
        break;
    }
    case Epi::Store:
    case Epi::StoreAdd: {
        float *out = ep.out0 + m0r * ep.ld + n;
        const bool add = ep.kind == Epi::StoreAdd;
        for (int i = lane >> 3; i < rows; i += 4) {
            float4 v = *reinterpret_cast<const float4 *>(sb + epi_at(i, lane & 7));
            const int64_t o = int64_t(i) * ep.ld;
            if (add) {
                if (ep.add_bf16) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(ep.add) +
                                                                     m0r * ep.ld + n + o);
                    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
                    const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
                    v = v + make_float4(p.x, p.y, q.x, q.y);
                } else {
                    v = v + ld_stream4(static_cast<const float *>(ep.add) + m0r * ep.ld + n + o);
                }
            }
            st_stream4(out + o, v);
            if (ep.out_x) st4(static_cast<__nv_bfloat16 *>(ep.out_x) + m0r * ep.ld + n + o, v);
        }
        break;
    }
    case Epi::Partial: {
        float *out = ep.out0 + (int64_t(z) * M + m0r) * args.Nc + n;
        for (int i = lane >> 3; i < rows; i += 4) st4(out + int64_t(i) * args.Nc, *reinterpret_cast<const float4 *>(sb + epi_at(i, lane & 7)));
        break;
    }
    }
}

template <bool ABF, bool BBF, bool SPLIT>
__global__ void __launch_bounds__(TC_THREADS_P, 1) k_gemm_tc(const TcArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int BN = args.BN, S = args.stages;
    const TcLayout Lo = tc_layout(BN, args.kper, args.b_res, SPLIT);
    uint8_t *bres = base;                                         // resident B (hi k-blocks, then lo)
    uint8_t *stages = base + Lo.bres_bytes;                       // ring of A (+B) stages
    float *esm = reinterpret_cast<float *>(stages + size_t(S) * Lo.stage_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(esm) + TC_EPI_SMEM);
    uint64_t *full = bars, *empty = bars + S, *accf = bars + 2 * S, *acce = bars + 2 * S + 2, *bready = bars + 2 * S + 4;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 5);
    volatile int *abort = reinterpret_cast<volatile int *>(bars + 2 * S + 5) + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = int64_t(args.n_tiles) * args.m_tiles * args.splits;
    const int64_t nkb_full = (args.kper + TC_BK - 1) / TC_BK;
    uint32_t ncols = 32;
    while (ncols < uint32_t(2 * BN)) ncols <<= 1;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), TC_PROD);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            mbar_init(smem_u32(&acce[b]), TC_EPI_WARPS * 32);
        }
        mbar_init(smem_u32(bready), TC_PROD);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == TC_MMA_WARP) {
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

    // tile t -> (z, m tile, n tile); k range of split z
    auto tile_of = [&](int64_t t, int64_t &m0, int64_t &n0, int &z, int64_t &kb0, int64_t &ke) {
        const int64_t per_split = int64_t(args.n_tiles) * args.m_tiles;
        z = int(t / per_split);
        const int64_t r = t - int64_t(z) * per_split;
        m0 = (r / args.n_tiles) * TC_BM;
        n0 = (r % args.n_tiles) * BN;
        kb0 = int64_t(z) * args.kper;
        ke = kb0 + args.kper < args.K ? kb0 + args.kper : args.K;
    };

    if (warp >= TC_EPI_WARPS && warp < TC_MMA_WARP) {
        // ---------------- producers
        const int ptid = tid - TC_EPI_WARPS * 32;
        bool ok = true;
        if (args.b_res) {
            // the n tile is the same for every tile of this CTA
            int64_t m0, n0, kb0, ke;
            int z;
            tile_of(blockIdx.x, m0, n0, z, kb0, ke);
            for (int64_t kb = 0; kb < nkb_full; ++kb) {
                uint8_t *hi = bres + size_t(kb) * Lo.b_bytes;
                uint8_t *lo = SPLIT ? bres + size_t(nkb_full + kb) * Lo.b_bytes : nullptr;
                stage_tile<BBF, SPLIT, false>(args.Bm, n0, args.Nc, BN, kb0 + kb * TC_BK, ke, hi, lo, ptid);
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(bready));
        }
        int64_t kbg = 0;   // k-blocks staged so far (ring position)
        for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            int64_t m0, n0, kb0, ke;
            int z;
            tile_of(t, m0, n0, z, kb0, ke);
            const int64_t nkb = ke > kb0 ? (ke - kb0 + TC_BK - 1) / TC_BK : 0;
            for (int64_t kb = 0; kb < nkb; ++kb, ++kbg) {
                const int s = int(kbg % S);
                const int64_t r = kbg / S;
                if (r > 0 && !mbar_wait(smem_u32(&empty[s]), uint32_t((r - 1) & 1), abort, args.status)) {
                    ok = false;
                    break;
                }
                uint8_t *st = stages + size_t(s) * Lo.stage_bytes;
                const uint32_t half = Lo.stage_bytes / (SPLIT ? 2 : 1);
                const int64_t k0 = kb0 + kb * TC_BK;
                stage_tile<ABF, SPLIT, true>(args.A, m0, args.M, TC_BM, k0, ke, st, SPLIT ? st + half : nullptr, ptid);
                if (!args.b_res)
                    stage_tile<BBF, SPLIT, false>(args.Bm, n0, args.Nc, BN, k0, ke, st + Lo.a_bytes,
                                                  SPLIT ? st + half + Lo.a_bytes : nullptr, ptid);
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&full[s]));
            }
        }
    } else if (warp == TC_MMA_WARP) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(BN);
            bool ok = !args.b_res || mbar_wait(smem_u32(bready), 0, abort, args.status);
            if (ok) tc_fence_after();
            int64_t kbg = 0, i = 0;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++i) {
                int64_t m0, n0, kb0, ke;
                int z;
                tile_of(t, m0, n0, z, kb0, ke);
                const int64_t nkb = ke > kb0 ? (ke - kb0 + TC_BK - 1) / TC_BK : 0;
                const int buf = int(i & 1);
                const int64_t ru = i >> 1;
                if (ru > 0 && !mbar_wait(smem_u32(&acce[buf]), uint32_t((ru - 1) & 1), abort, args.status)) break;
                tc_fence_after();
                const uint32_t dacc = tmem + uint32_t(buf * BN);
                for (int64_t kb = 0; kb < nkb; ++kb, ++kbg) {
                    const int s = int(kbg % S);
                    const int64_t r = kbg / S;
                    if (!mbar_wait(smem_u32(&full[s]), uint32_t(r & 1), abort, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(stages + size_t(s) * Lo.stage_bytes);
                    const uint32_t half = Lo.stage_bytes / (SPLIT ? 2 : 1);
                    const uint32_t a_hi = st, a_lo = st + half;
                    uint32_t b_hi, b_lo;
                    if (args.b_res) {
                        b_hi = smem_u32(bres + size_t(kb) * Lo.b_bytes);
                        b_lo = smem_u32(bres + size_t(nkb_full + kb) * Lo.b_bytes);
                    } else {
                        b_hi = st + Lo.a_bytes;
                        b_lo = st + half + Lo.a_bytes;
                    }
#pragma unroll
                    for (int ks = 0; ks < TC_BK / 16; ++ks) {
                        const uint32_t koff = uint32_t(ks) * 32u;
                        const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
                        mma_bf16(dacc, sw128_desc(a_hi + koff), sw128_desc(b_hi + koff), idesc, acc);
                        if (SPLIT) {
                            mma_bf16(dacc, sw128_desc(a_hi + koff), sw128_desc(b_lo + koff), idesc, 1u);
                            mma_bf16(dacc, sw128_desc(a_lo + koff), sw128_desc(b_hi + koff), idesc, 1u);
                        }
                    }
                    mma_commit(smem_u32(&empty[s]));
                }
                mma_commit(smem_u32(&accf[buf]));
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warp w: TMEM lanes 32*(w%4).., columns of half w/4)
        float *sb = esm + warp * (32 * 32);
        const int q = warp & 3, half = warp >> 2;
        int64_t i = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            int64_t m0, n0, kb0, ke;
            int z;
            tile_of(t, m0, n0, z, kb0, ke);
            const int64_t nkb = ke > kb0 ? (ke - kb0 + TC_BK - 1) / TC_BK : 0;
            const int buf = int(i & 1);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&accf[buf]), uint32_t((i >> 1) & 1), abort, args.status));
            tc_fence_after();
            const int64_t m0r = m0 + q * 32;
            for (int c = half * 32; c < BN; c += 64) {
                float v[32];
                if (ok && nkb > 0) {
                    tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(buf * BN + c), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(sb + epi_at(lane, j >> 2)) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                __syncwarp();
                if (m0r < args.M) epi_chunk(args, sb, m0r, int(n0) + c, z, lane);
                __syncwarp();
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&acce[buf]));
            if (!ok) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == TC_MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

// ---------------------------------------------------------------- launcher
static int g_num_sms = 0;

template <bool ABF, bool BBF, bool SPLIT>
static cudaError_t launch_tc_t(const TcArgs &a, unsigned grid, size_t smem, cudaStream_t st) {
    auto kern = k_gemm_tc<ABF, BBF, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, TC_THREADS_P, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tc(int64_t M, int64_t Nc, int64_t K, const GemmOperand &A, const GemmOperand &Bm,
                           const GemmEpilogue &ep, int splits, bool split3, unsigned *status, cudaStream_t st) {
    if (M <= 0 || Nc <= 0) return cudaSuccess;
    if (splits < 1) splits = 1;
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    TcArgs a;
    a.M = M; a.Nc = Nc; a.K = K; a.splits = splits;
    int64_t kper = (K + splits - 1) / splits;
    a.kper = (kper + TC_BK - 1) / TC_BK * TC_BK;
    // Tile width: the widest (<= 256, a multiple of 32) whose stages fit; B resident when its
    // whole k extent fits next to two A stages and the epilogue buffer.
    const size_t budget = 227 * 1024 - 1024 - TC_EPI_SMEM - 256;
    int BN = int(Nc < 256 ? (Nc + 31) / 32 * 32 : 256);
    int S = 0;
    for (;; BN = BN > 32 ? (BN / 2 + 31) / 32 * 32 : 0) {
        if (BN == 0) return cudaErrorInvalidConfiguration;
        const TcLayout res = tc_layout(BN, a.kper, true, split3);
        a.b_res = splits == 1 && size_t(res.bres_bytes) + 2 * size_t(res.stage_bytes) <= budget;
        const TcLayout Lt = tc_layout(BN, a.kper, a.b_res, split3);
        S = int((budget - Lt.bres_bytes) / Lt.stage_bytes);
        if (S >= 2) break;
    }
    if (S > 6) S = 6;
    a.BN = BN;
    a.stages = S;
    a.n_tiles = int((Nc + BN - 1) / BN);
    a.m_tiles = int((M + TC_BM - 1) / TC_BM);
    a.A = A; a.Bm = Bm; a.ep = ep; a.status = status;
    const TcLayout L = tc_layout(BN, a.kper, a.b_res, split3);
    const size_t smem = 1024 + size_t(L.bres_bytes) + size_t(S) * L.stage_bytes + TC_EPI_SMEM + (2 * S + 6) * 8;
    const int64_t ntiles = int64_t(a.n_tiles) * a.m_tiles * splits;
    int64_t grid = ntiles;
    if (grid > g_num_sms) grid = (g_num_sms / a.n_tiles) * a.n_tiles;
    if (grid < a.n_tiles) grid = a.n_tiles;
    if (grid > ntiles) grid = ntiles;
    if (split3) {
        if (A.bf16 && Bm.bf16) return launch_tc_t<true, true, true>(a, unsigned(grid), smem, st);
        if (A.bf16) return launch_tc_t<true, false, true>(a, unsigned(grid), smem, st);
        if (Bm.bf16) return launch_tc_t<false, true, true>(a, unsigned(grid), smem, st);
        return launch_tc_t<false, false, true>(a, unsigned(grid), smem, st);
    }
    if (A.bf16 && Bm.bf16) return launch_tc_t<true, true, false>(a, unsigned(grid), smem, st);
    if (A.bf16) return launch_tc_t<true, false, false>(a, unsigned(grid), smem, st);
    if (Bm.bf16) return launch_tc_t<false, true, false>(a, unsigned(grid), smem, st);
    return launch_tc_t<false, false, false>(a, unsigned(grid), smem, st);
}

}  // namespace adj
