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
// CTA: 18 warps in four roles (epilogue, producers, MMA issuer, TMA issuer; see the
// kernel below).  Stages, accumulators and the resident B tile are handed over with
// mbarriers, and every wait is bounded by a wall-clock limit.
//
// Tile: BM = 128 rows (TMEM lanes), BN <= 256 columns (TMEM columns), BK = 64
// (one 128-byte swizzle row of bf16).  Shared-memory element (r, k) of a tile lives
// at byte r*128 + ((k/8) ^ (r%8))*16 + (k%8)*2 (8-row atoms of 1024 bytes).
#include <stdlib.h>
#include <string.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "adj_internal.cuh"
#include "adj_epilogue.cuh"
#include "adj_ptx.cuh"
#include "adj_tmap.cuh"

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
// Shared-memory matrix descriptor: MN-major, 128-byte swizzle.  The tile is stored as
// blocks of 64 M (or N) elements x 64 k rows (8 KB, one TMA box each): 128-byte rows of
// 64 elements, 8-row groups 1024 B apart (stride byte offset), 64-element blocks 8 KB
// apart (leading byte offset).  One MMA k-step of 16 rows advances the start by 2 KB.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t(8192 >> 4) << 16;
    d |= uint64_t(1024 >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}
// Instruction descriptor: kind::f16, bf16 x bf16 -> fp32; a_mn / b_mn select MN-major operands.
__device__ __forceinline__ uint32_t idesc_bf16(int n, bool a_mn = false, bool b_mn = false, int m = TC_BM) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
           (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
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
// CTA pair: one MMA over both CTAs' operands (A: 128 rows in each CTA; B: half the
// columns in each), D in both CTAs' tensor memory at the same address.
__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// CTA pair: arrive on the mbarrier at this shared-memory offset in both CTAs once the
// pair MMAs issued so far have completed
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask = 3) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
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

// Low-part array of the array p of a pre-split operand.
__device__ __forceinline__ const void *lo_of(const GemmOperand &O, const void *p) {
    return p == O.p[0] ? O.lo[0] : p == O.p[1] ? O.lo[1] : O.lo[2];
}

// Stage rows [row0, row0+R) x k [k0, k0+64) of an operand into a swizzled tile.  A
// pre-split operand is staged as hi + lo (and split again in split mode).
// k-contiguous sources: a work item is 8 consecutive k of one row (two float4 or one
// 16-byte bf16 vector).  Row-contiguous sources (the token-major operands of the
// parameter reductions): a work item is a 4-row (fp32) or 8-row (bf16) by 8-k block,
// loaded as 8 row vectors and transposed in registers.  Loads of a thread's items are
// issued before any is converted, so several vectors are in flight per thread.
template <bool BF, bool SPLIT, bool IS_A>
__device__ __forceinline__ void stage_tile(const GemmOperand &O, int64_t row0, int64_t rows, int R, int64_t k0,
                                           int64_t kend, uint8_t *hi, uint8_t *lo, int tid) {
    constexpr int BATCH = 2;
    // vector loads need every row (k-contiguous source) or every k row (row-contiguous
    // source) to start on a 16-byte boundary; other strides take the element-wise path
    const bool kvec = O.s_row % (BF ? 8 : 4) == 0;
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
                    if (k + 8 <= kend && kvec) {
                        ld8_contig<BF>(p, i, v[b]);
                        if (BF && O.lo[0]) {
                            float l[8];
                            ld8_contig<true>(lo_of(O, p), i, l);
#pragma unroll
                            for (int j = 0; j < 8; ++j) v[b][j] += l[j];
                        }
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
                            if (BF && O.lo[0] && k + j < kend) v[b][j] += ld1<true>(lo_of(O, p), i + j);
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
        const bool full = row + RB <= rows && k + 8 <= kend && O.s_k % RB == 0;
        if (BF && full) {
            // 8 k rows of 8 bf16 each, kept packed (and the low parts of a pre-split
            // operand), unpacked one output row at a time
            uint4 u[8], ul[8];
            const bool pre = O.lo[0] != nullptr;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int64_t i;
                const void *p = op_at<IS_A>(O, row, k + j, i);
                u[j] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + i));
                ul[j] = pre ? __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(lo_of(O, p)) + i))
                            : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t w = (&u[j].x)[q >> 1], wl = (&ul[j].x)[q >> 1];
                    v[j] = __uint_as_float((q & 1) ? (w & 0xFFFF0000u) : (w << 16)) +
                           __uint_as_float((q & 1) ? (wl & 0xFFFF0000u) : (wl << 16));
                }
                put8<SPLIT>(hi, lo, r0 + q, kc, v);
            }
            continue;
        }
        float v[RB][8];   // v[row][k]
        if (!BF && full) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int64_t i;
                const void *p = op_at<IS_A>(O, row, k + j, i);
                const float4 f = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
                v[0][j] = f.x; v[1 % RB][j] = f.y; v[2 % RB][j] = f.z; v[3 % RB][j] = f.w;
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
                        if (BF && O.lo[0]) x += ld1<true>(lo_of(O, p), i);
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
//   warp 17     lane 0 issues the TMA tile loads, running ahead of the producers by up to
//               S stages (bf16 tiles land in the MMA layout; fp32 tiles land raw and the
//               producers convert them in place)
// Barriers: full[s]/empty[s] hand stages producer -> MMA -> producer; accf[b]/acce[b]
// hand accumulator b MMA -> epilogue -> MMA; bres marks the resident B tile ready.
#ifndef ADJ_TC_EPI_WARPS
#define ADJ_TC_EPI_WARPS 8
#endif
constexpr int TC_EPI_WARPS = ADJ_TC_EPI_WARPS, TC_THREADS_P = (TC_EPI_WARPS + TC_PROD_WARPS + 2) * 32;
static_assert(TC_EPI_WARPS % 4 == 0, "epilogue warps cover the four TMEM lane quarters");
constexpr int TC_MMA_WARP = TC_EPI_WARPS + TC_PROD_WARPS, TC_TMA_WARP = TC_MMA_WARP + 1;
constexpr uint32_t TC_EPI_SMEM = TC_EPI_WARPS * 32 * 32 * 4;
// CTA pairs need no producer warps (every operand comes by TMA): a pair kernel with many
// tiles per CTA runs warps 0-15 as epilogue warps, twice the output chunks in flight
constexpr int TC_MAX_EPI_WARPS = TC_EPI_WARPS + TC_PROD_WARPS;
constexpr uint32_t TC_CHUNK_BYTES = 32 * 32 * 4;
// A streamed StoreAdd pair product with a short K (the output projection) can keep each CTA's
// half of the B tile resident (TC_RO_BRES) and stream only A through TC_RO_STAGES stages; the
// shared memory that frees gives TC_RO_EPI_WARPS epilogue warps a residual buffer and an
// output buffer each.  16 warps with two A stages measured best (12 warps with four stages, or
// three streamed A+B stages without the resident B, were slower)
#ifndef ADJ_TC_RO_EPI_WARPS
#define ADJ_TC_RO_EPI_WARPS 16
#endif
#ifndef ADJ_TC_RO_STAGES
#define ADJ_TC_RO_STAGES 2
#endif
#ifndef ADJ_TC_RO_BRES
#define ADJ_TC_RO_BRES 1
#endif
constexpr int TC_RO_EPI_WARPS = ADJ_TC_RO_EPI_WARPS, TC_RO_STAGES = ADJ_TC_RO_STAGES;
constexpr bool TC_RO_BRES = ADJ_TC_RO_BRES;

// Operand load mode: register staging, or TMA tiles of a bf16 array (K-major: one box of
// 64 k x R rows; MN-major: R/64 boxes of 64 rows x 64 k).
enum { LD_REG = 0, LD_TMA_K = 1, LD_TMA_MN = 2, LD_RAW_K = 3, LD_RAW_MN = 4 };
__host__ __device__ inline bool ld_raw(int m) { return m >= LD_RAW_K; }
__host__ __device__ inline bool ld_tma(int m) { return m != LD_REG; }

// Four-CTA clusters (two pairs on the same n tile and neighbouring m tiles): a 2-D tiled TMA
// load multicast to the CTAs of `mask` (the same shared offset in each); each destination's
// completion is counted on the mbarrier at `bar`'s offset in the leader CTA of that
// destination's pair (bar: the issuing pair's leader barrier, peer bit clear).
__device__ __forceinline__ void tma_load_2d_quad(uint32_t dst, const void *tmap, int x, int y, uint32_t bar,
                                                 uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "h"(mask)
        : "memory");
}

// Advance a ring position (slot s of S, round r) by one stage, without a 64-bit division in
// the hot loops of the single-thread TMA and MMA issuers.
__device__ __forceinline__ void ring_next(int &s, int64_t &r, int S) {
    if (++s == S) {
        s = 0;
        ++r;
    }
}

// L2 priorities for a streamed StoreAdd epilogue: the outputs and the consumed residual and
// xhat lines are marked evict-first, so that the boxes prefetched a tile ahead are not the
// ones pushed out of L2 by the output stream.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void *tmap, int x, int y, uint32_t bar,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d_hint(const void *tmap, int x, int y, uint32_t src, uint64_t pol) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(src), "l"(pol)
                 : "memory");
}

struct TcArgs {
    CUtensorMap tmA[3], tmB[3];   // one map per array of a blocked operand
    CUtensorMap tmBlo[3];         // low parts of a pre-split B
    CUtensorMap tmAmul;           // the elementwise factor of a raw-loaded A
    CUtensorMap tmO[3];           // epilogue outputs stored by TMA (ProjIn: a, u, c)
    CUtensorMap tmAdd;            // StoreAdd: the residual, loaded by TMA
    CUtensorMap tmNx;             // StoreAdd through a normalised input: xhat, prefetched into L2
    int64_t M, Nc, K, kper;
    int BN, stages, n_tiles, m_tiles, splits;
    int a_ld, b_ld;
    bool b_res, a_mul, b_lo;
    bool epi_tma;                 // epilogue through TMA stores (tmO, tmAdd)
    bool stream_out;              // StoreAdd whose output far exceeds L2: evict-first hints
    bool ro;                      // streamed StoreAdd with separate residual and output buffers
    bool add16;                   // StoreAdd residual in bf16 by TMA (32 x 32 boxes, dense 64-byte rows)
    bool outx_tma;                // the bf16 copy (out_x) staged per warp and stored by TMA
    bool nx_tma;                  // (with outx_tma) the bf16 normalised input loaded into that buffer by TMA
    CUtensorMap tmOx;             // out_x: 32 x 32 bf16 boxes, unswizzled
    CUtensorMap tmNxl;            // nx (bf16) for loads: the same box shape
    int nacc;                     // accumulators in tensor memory (2: epilogue overlaps the next tile)
    int epiw;                     // epilogue warps (CTA pairs: 8 or 16; otherwise TC_EPI_WARPS)
    GemmOperand A, Bm;
    GemmEpilogue ep;
    unsigned *status;
};

// Issue the TMA loads of rows [row0, row0+R) x k [k0, k0+64) of an operand into dst.
template <bool IS_A, bool PAIRLD = false>
__device__ __forceinline__ void tma_tile(const CUtensorMap *maps, const GemmOperand &O, int mode, int64_t row0, int R,
                                         int64_t k0, uint8_t *dst, uint32_t bar) {
    int blk = 0;
    int64_t rr = row0, kk = k0;
    if (O.blk < (int64_t(1) << 30)) {
        if (IS_A) {
            blk = int(k0 / O.blk);
            kk = k0 - int64_t(blk) * O.blk;
        } else {
            blk = int(row0 / O.blk);
            rr = row0 - int64_t(blk) * O.blk;
        }
    }
    const void *m = &maps[blk];
    if (mode == LD_TMA_K || mode == LD_RAW_K) {
        if (PAIRLD) tma_load_2d_pair(smem_u32(dst), m, int(kk), int(rr), bar);
        else tma_load_2d(smem_u32(dst), m, int(kk), int(rr), bar);
    } else {
        const int box = mode == LD_RAW_MN ? 16384 : 8192;   // 64 x 64 fp32 or bf16
        for (int j = 0; j < R / 64; ++j) {
            if (PAIRLD) tma_load_2d_pair(smem_u32(dst + j * box), m, int(rr) + 64 * j, int(kk), bar);
            else tma_load_2d(smem_u32(dst + j * box), m, int(rr) + 64 * j, int(kk), bar);
        }
    }
}

// Convert a raw fp32 tile (R = 128 rows x 64 k, as TMA wrote it) in place into the bf16
// hi (and lo) tiles of the swizzled K-major layout.  Raw layouts: k-contiguous source:
// row r at r*256 B; row-contiguous source: boxes of 64 rows, box j at j*16 KB holding
// [k][row] with 256-byte k rows.  Every producer thread reads all its values first, the
// producers meet at a named barrier, then write (hi at region, lo at region + 16 KB).
// Both mappings keep shared-memory reads and writes free of bank conflicts: k-contiguous
// tiles are read as 16-byte vectors, 32 lanes covering two full rows, and written as
// 8-byte halves of the swizzled 16-byte chunks; row-contiguous tiles are read one value
// per lane (32 consecutive rows) and written as whole chunks of one row per lane.
__device__ __forceinline__ void put4(uint8_t *hi, uint8_t *lo, int r, int k4, float4 v, bool split) {
    const uint32_t off = uint32_t(r) * 128u + (uint32_t((k4 >> 1) ^ (r & 7)) << 4) + uint32_t(k4 & 1) * 8u;
    uint2 h;
    h.x = pack_bf16(v.x, v.y);
    h.y = pack_bf16(v.z, v.w);
    *reinterpret_cast<uint2 *>(hi + off) = h;
    if (split) {
        uint2 l;
        l.x = pack_bf16(v.x - bf16_round(v.x), v.y - bf16_round(v.y));
        l.y = pack_bf16(v.z - bf16_round(v.z), v.w - bf16_round(v.w));
        *reinterpret_cast<uint2 *>(lo + off) = l;
    }
}

// With csum (row-contiguous tiles only) it returns the sum, in a fixed order, of the raw
// values of the thread's row r = ptid % 128 (column sums of a token-major operand); else 0.
template <bool SPLIT, bool MN, bool MUL = false, int NP = TC_PROD>
__device__ __forceinline__ float convert_raw128(uint8_t *region, int ptid, bool csum = false) {
    float rsum = 0.f;
    constexpr int R = TC_BM;
    const float *raw = reinterpret_cast<const float *>(region);
    if (!MN) {
        constexpr int ITEMS = R * 16, PER = (ITEMS + NP - 1) / NP;   // float4 (4 k of one row)
        float4 v[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int q = ptid + i * NP;
            if (ITEMS % NP == 0 || q < ITEMS) v[i] = reinterpret_cast<const float4 *>(raw)[q];
        }
        if (MUL) {
            // the factor tile (same layout) follows the operand tile
            const float4 *mraw = reinterpret_cast<const float4 *>(region + R * 256);
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int q = ptid + i * NP;
                if (ITEMS % NP == 0 || q < ITEMS) v[i] = v[i] * mraw[q];
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NP) : "memory");
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int q = ptid + i * NP;    // float4 index: row q/16, k4 q%16
            if (ITEMS % NP == 0 || q < ITEMS) put4(region, region + R * 128, q >> 4, q & 15, v[i], SPLIT);
        }
    } else {
        constexpr int ITEMS = R * 8, PER = (ITEMS + NP - 1) / NP;    // items (one row, 8 k)
        float v[PER][8];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int it = ptid + i * NP, r = it % R, kc = it / R;
            const float *src = raw + (r >> 6) * 4096 + (r & 63);
            if (ITEMS % NP == 0 || it < ITEMS) {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[i][j] = src[(kc * 8 + j) * 64];
            }
        }
        if (csum) {
            static_assert(NP % R == 0, "a thread keeps one row");
#pragma unroll
            for (int i = 0; i < PER; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) rsum += v[i][j];
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NP) : "memory");
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int it = ptid + i * NP;
            if (ITEMS % NP == 0 || it < ITEMS) put8<SPLIT>(region, region + R * 128, it % R, it / R, v[i]);
        }
    }
    return rsum;
}

// Shared-memory layout.  A stage holds the A region then (unless B is resident) the B
// region.  A region: bf16 hi tile, then the lo tile (split mode); an operand loaded raw
// (fp32 by TMA, converted in place) needs twice the bf16 tile, which the split mode's
// hi + lo already provides, and a raw operand with an elementwise factor twice that
// again (the factor's raw tile follows).  Resident B: per k-block a hi tile then a lo tile.
struct TcLayout {
    uint32_t a_bytes, b_bytes, a_reg, b_reg, stage_bytes, bres_kb, bres_bytes;
};
__host__ __device__ inline TcLayout tc_layout(int BN, int64_t K, bool b_res, bool split, bool a_raw = false,
                                              bool b_raw = false, bool a_mul = false) {
    TcLayout L;
    const uint32_t f = split ? 2u : 1u;
    L.a_bytes = TC_BM * 128u;
    L.b_bytes = uint32_t(BN) * 128u;
    L.a_reg = L.a_bytes * (a_mul ? 4u : (split || a_raw) ? 2u : 1u);
    L.b_reg = b_res ? 0u : L.b_bytes * ((split || b_raw) ? 2u : 1u);
    L.stage_bytes = L.a_reg + L.b_reg;
    const uint32_t kb = uint32_t((K + TC_BK - 1) / TC_BK);
    L.bres_kb = L.b_bytes * f;
    L.bres_bytes = b_res ? L.bres_kb * kb : 0u;
    return L;
}

// Epilogue of one 32-row x 32-column chunk held in shared memory: row r, column quad q
// (columns 4q..4q+3) at float offset r*32 + 4*(q ^ (r%8)) (conflict-free both ways).
// Lane l owns quad l%8 of rows l/8, l/8+4, ...: every store is a 16-byte vector and a
// warp writes four full 128-byte row segments per instruction.
__device__ __forceinline__ int epi_at(int r, int q) { return r * 32 + ((q ^ (r & 7)) << 2); }

__device__ __forceinline__ float sigmoidf_fast(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// EXT: the epilogue features only some launches use (the cotangent through a normalised
// input, a lane-written bf16 copy of the output in the TMA path) are compiled in; the other
// instantiations leave them out, which keeps their register use (and spills) down.
template <bool EXT>
__device__ __forceinline__ void epi_chunk(const TcArgs &args, const float *sb, int64_t m0r, int n0c, int z, int lane) {
    const GemmEpilogue &ep = args.ep;
    const int64_t M = args.M;
    const int cq = (lane & 7) * 4, n = n0c + cq;
    if (n >= args.Nc) return;                    // Nc is a multiple of 8: a column quad is all in or all out
    const int rows = M - m0r < 32 ? int(M - m0r) : 32;
    switch (ep.kind) {
    case Epi::ProjIn: {
        int blk, j;
        projin_col(ep, n, blk, j);
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
            if (EXT && add && ep.nr) {
                // through the normalised input: (acc - xhat mean(xhat . dxhat)) / r, then the add
                const int64_t row = m0r + i;
                float sdz = 0.f;
                for (int sl = 0; sl < ep.nsl; ++sl) sdz += __ldg(ep.ndz + row * ep.nsl + sl);
                const float mt = sdz * ep.inv_P, ir = 1.f / __ldg(ep.nr + row);
                float4 x4;
                if (ep.nx_bf16) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(ep.nx) + row * ep.ld + n);
                    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
                    const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
                    x4 = make_float4(p.x, p.y, q.x, q.y);
                } else {
                    x4 = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(ep.nx) + row * ep.ld + n));
                }
                v = (v - x4 * f4(mt)) * f4(ir);
            }
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

// REGS: whether register staging may be needed (any operand with LD_REG, or a resident B
// not loaded by TMA).  Without it the kernel carries no staging code, which keeps the
// producers' hot loop free of register spills; ABF/BBF only matter with REGS.
// PAIR: the kernel runs as clusters of two CTAs on neighbouring SMs.  A pair computes a
// 256-row x BN tile with one tcgen05.mma.cta_group::2 per k-slice: each CTA stages its
// 128 rows of A and half of the B tile (BN / 2 output columns) by TMA, both CTAs' loads
// complete on the leader's (rank 0) stage barrier, the leader issues the MMAs, and the
// accumulator (128 rows per CTA) lands in both CTAs' tensor memory.  The MMA completion
// is multicast to both CTAs' stage and accumulator barriers; both epilogues release the
// accumulator on the leader's barrier.  Per SM this halves the B operand traffic through
// shared memory for the same MMA work.  Only all-bf16, all-TMA operands take this mode.
// QUAD (with PAIR): clusters of four CTAs, two pairs on the same n tile and the two halves
// of a 512-row m tile.  The pairs' B halves are the same: each CTA loads half of its B half
// and multicasts it to its counterpart in the other pair, so B crosses L2 once per four
// CTAs instead of twice.  A stage is refilled only once both pairs' MMAs have released it.
template <bool ABF, bool BBF, bool SPLIT, bool REGS, bool PAIR = false, bool EXT = false, bool QUAD = false>
__global__ void __launch_bounds__(TC_THREADS_P, 1) k_gemm_tc(const __grid_constant__ TcArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int BN = args.BN, S = args.stages;
    const int BNS = PAIR ? BN / 2 : BN;   // B rows (output columns) staged by this CTA
    const TcLayout Lo = tc_layout(BNS, args.kper, args.b_res, SPLIT, ld_raw(args.a_ld), ld_raw(args.b_ld), args.a_mul);
    uint8_t *bres = base;                                         // resident B (hi k-blocks, then lo)
    uint8_t *stages = base + Lo.bres_bytes;                       // ring of A (+B) stages
    const int EPIW = PAIR ? args.epiw : TC_EPI_WARPS;
    float *esm = reinterpret_cast<float *>(stages + size_t(S) * Lo.stage_bytes);
    // (ro) EPIW output chunk buffers, (outx_tma) then EPIW bf16 chunk buffers of 2 KB
    // only a pair kernel (no quad) without the EXT epilogue features is launched with ro, and
    // only a pair kernel without them with a bf16 residual by TMA
    const bool RO = PAIR && !QUAD && !EXT && args.ro;
    const bool ADD16 = PAIR && !EXT && args.add16;
    const uint32_t add_tx = ADD16 ? 32u * 32u * 2u : 32u * 32u * 4u;   // residual bytes a chunk
    const size_t ro_bytes = RO ? size_t(EPIW) * TC_CHUNK_BYTES : 0;
    uint16_t *esx =
        reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(esm) + size_t(EPIW) * TC_CHUNK_BYTES + ro_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(esm) + size_t(EPIW) * TC_CHUNK_BYTES +
                                                  ro_bytes + (args.outx_tma ? size_t(EPIW) * TC_CHUNK_BYTES / 2 : 0));
    uint64_t *full = bars, *empty = bars + S, *accf = bars + 2 * S, *acce = bars + 2 * S + 2, *bready = bars + 2 * S + 4;
    uint64_t *rawfull = bars + 2 * S + 5, *addb = bars + 3 * S + 5;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bars + 3 * S + 5 + TC_MAX_EPI_WARPS);
    volatile int *abort = reinterpret_cast<volatile int *>(bars + 3 * S + 5 + TC_MAX_EPI_WARPS) + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = int64_t(args.n_tiles) * args.m_tiles * args.splits;
    const int64_t nkb_full = (args.kper + TC_BK - 1) / TC_BK;
    // tiles are scheduled per CTA, or per pair (unit = cluster) with rank 0 the leader; a
    // four-CTA cluster holds pairs {0, 1} and {2, 3} (leaders 0 and 2)
    const uint32_t crank = PAIR ? cluster_rank() : 0u;
    const uint32_t prank = crank & 1u, lead = crank & ~1u, pq = QUAD ? crank >> 1 : 0u;
    const int64_t unit0 = QUAD ? int64_t(blockIdx.x >> 2) : PAIR ? int64_t(blockIdx.x >> 1) : int64_t(blockIdx.x);
    const int64_t nunits = QUAD ? int64_t(gridDim.x >> 2) : PAIR ? int64_t(gridDim.x >> 1) : int64_t(gridDim.x);
    const int NACC = PAIR ? args.nacc : 2;
    uint32_t ncols = 32;
    while (ncols < uint32_t(NACC * BN)) ncols <<= 1;
    // who fills a stage: the producers (register staging or in-place conversion of raw
    // tiles) and/or the TMA warp (bf16 tiles straight into the MMA layout)
    const bool b_here = !args.b_res;
    const bool a_raw = ld_raw(args.a_ld), b_raw = b_here && ld_raw(args.b_ld);
    const bool a_dir = ld_tma(args.a_ld) && !a_raw, b_dir = b_here && ld_tma(args.b_ld) && !b_raw;
    const bool a_reg = args.a_ld == LD_REG, b_reg = b_here && args.b_ld == LD_REG;
    const bool prod_full = a_reg || b_reg || a_raw || b_raw, tma_full = a_dir || b_dir;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), (prod_full ? TC_PROD : 0) + (tma_full ? 1 : 0));
            mbar_init(smem_u32(&empty[s]), QUAD ? 2 : 1);   // QUAD: both pairs' MMAs release the stage
            mbar_init(smem_u32(&rawfull[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            // CTA pair: one arrival per epilogue warp of both CTAs, on the leader's barrier
            mbar_init(smem_u32(&acce[b]), PAIR ? 2 * EPIW : EPIW * 32);
        }
        mbar_init(smem_u32(bready), ld_tma(args.b_ld) ? 1 : TC_PROD);
        for (int w = 0; w < EPIW; ++w) mbar_init(smem_u32(&addb[w]), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == TC_MMA_WARP) {
        if (PAIR) {
            // one warp of each CTA of the pair allocates, collectively, in both SMs
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(const_cast<uint32_t *>(tmem_slot))),
                         "r"(ncols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(const_cast<uint32_t *>(tmem_slot))),
                         "r"(ncols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    if (PAIR) cluster_sync();   // also: the peer's barriers are initialised before any remote use
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // CTA pair: both CTAs must hold the accumulator at the same tensor-memory address (the
    // pair MMA writes it there in both); otherwise nothing runs and a failure is recorded
    bool pair_ok = true;
    if (PAIR) {
        const uint32_t peer = ld_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t *>(tmem_slot)), crank ^ 1u));
        pair_ok = peer == tmem;
        if (!pair_ok && tid == 0) record_timeout(args.status);
    }

    // tile t -> (z, m tile, n tile); k range of split z
    auto tile_of = [&](int64_t t, int64_t &m0, int64_t &n0, int &z, int64_t &kb0, int64_t &ke) {
        const int64_t per_split = int64_t(args.n_tiles) * args.m_tiles;
        z = int(t / per_split);
        const int64_t r = t - int64_t(z) * per_split;
        m0 = (r / args.n_tiles) * (QUAD ? 4 * TC_BM : PAIR ? 2 * TC_BM : TC_BM) + int64_t(pq) * 2 * TC_BM +
             int64_t(prank) * TC_BM;   // this CTA's rows
        n0 = (r % args.n_tiles) * BN;
        kb0 = int64_t(z) * args.kper;
        ke = kb0 + args.kper < args.K ? kb0 + args.kper : args.K;
    };

    if (warp >= EPIW && warp < TC_MMA_WARP) {
        // ---------------- producers
        const int ptid = tid - TC_EPI_WARPS * 32;
        bool ok = true;
        if constexpr (REGS) if (args.b_res && !ld_tma(args.b_ld)) {
            // the n tile is the same for every tile of this CTA
            int64_t m0, n0, kb0, ke;
            int z;
            tile_of(blockIdx.x, m0, n0, z, kb0, ke);
            for (int64_t kb = 0; kb < nkb_full; ++kb) {
                uint8_t *hi = bres + size_t(kb) * Lo.bres_kb;
                uint8_t *lo = SPLIT ? hi + Lo.b_bytes : nullptr;
                stage_tile<BBF, SPLIT, false>(args.Bm, n0, args.Nc, BN, kb0 + kb * TC_BK, ke, hi, lo, ptid);
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(bready));
        }
        const bool any_raw = a_raw || b_raw;
        // column sums of B's first ep.csum_n columns (the raw row-contiguous B of a
        // one-tile-per-CTA split-K product): row ptid % 128 of each 128-row half
        const bool csum_on = args.ep.csum && b_raw && args.b_ld == LD_RAW_MN && args.ep.kind == Epi::Partial;
        float csum0 = 0.f, csum1 = 0.f;
        int64_t kbg = 0;   // k-blocks staged so far (ring position)
        int rs = 0;        // its slot and round
        int64_t rr = 0;
        for (int64_t t = unit0; t < ntiles && ok && prod_full; t += nunits) {
            int64_t m0, n0, kb0, ke;
            int z;
            tile_of(t, m0, n0, z, kb0, ke);
            const int64_t nkb = ke > kb0 ? (ke - kb0 + TC_BK - 1) / TC_BK : 0;
            for (int64_t kb = 0; kb < nkb; ++kb, ++kbg, ring_next(rs, rr, S)) {
                const int s = rs;
                const int64_t r = rr;
                uint8_t *st = stages + size_t(s) * Lo.stage_bytes;
                uint8_t *sa = st, *sbb = st + Lo.a_reg;
                const int64_t k0 = kb0 + kb * TC_BK;
                if constexpr (REGS) if (a_reg || b_reg) {
                    // register-staged tiles overwrite the stage: wait until the MMAs released it
                    bool got = r == 0 || mbar_wait(smem_u32(&empty[s]), uint32_t((r - 1) & 1), abort, args.status);
                    // with raw tiles the producers meet at named barriers, so they decide together
                    if (any_raw) got = bar_red_and(1, TC_PROD, got);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    if (a_reg)
                        stage_tile<ABF, SPLIT, true>(args.A, m0, args.M, TC_BM, k0, ke, sa,
                                                     SPLIT ? sa + Lo.a_bytes : nullptr, ptid);
                    if (b_reg)
                        stage_tile<BBF, SPLIT, false>(args.Bm, n0, args.Nc, BN, k0, ke, sbb,
                                                      SPLIT ? sbb + Lo.b_bytes : nullptr, ptid);
                }
                if (any_raw) {
                    // the raw tile of round r lands only after the MMAs released round r-1
                    if (!bar_red_and(1, TC_PROD, mbar_wait(smem_u32(&rawfull[s]), uint32_t(r & 1), abort, args.status))) {
                        ok = false;
                        break;
                    }
                    if (a_raw) {
                        if (args.a_ld == LD_RAW_MN) convert_raw128<SPLIT, true>(sa, ptid);
                        else if (args.a_mul) convert_raw128<SPLIT, false, true>(sa, ptid);
                        else convert_raw128<SPLIT, false>(sa, ptid);
                    }
                    if (b_raw) {
                        // a 256-row B tile converts as two independent 128-row halves
                        const bool bmn = args.b_ld == LD_RAW_MN;
                        int half = 0;
                        for (uint8_t *bh = sbb; bh < sbb + BN * 256; bh += 2 * TC_BM * 128, ++half) {
                            if (bmn) {
                                const float rs = convert_raw128<SPLIT, true>(bh, ptid, csum_on);
                                if (half == 0) csum0 += rs;
                                else csum1 += rs;
                            } else {
                                convert_raw128<SPLIT, false>(bh, ptid);
                            }
                        }
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&full[s]));
            }
        }
        if (csum_on && ok) {
            // this CTA's one tile: column n0 + 128 h + r; the two threads of a row hold the
            // even and the odd k chunks: partial [2 z + ptid / 128][n] for n < csum_n
            int64_t m0, n0, kb0, ke;
            int z;
            tile_of(blockIdx.x, m0, n0, z, kb0, ke);
            float *out = args.ep.csum + (2 * int64_t(z) + ptid / TC_BM) * args.ep.csum_n;
            const int64_t n = n0 + ptid % TC_BM;
            if (n < args.ep.csum_n) out[n] = csum0;
            if (BN > TC_BM && n + TC_BM < args.ep.csum_n) out[n + TC_BM] = csum1;
        }
    }
    if (warp == TC_TMA_WARP) {
        // ---------------- TMA issuer
        if (lane == 0) {
            if (args.b_res && ld_tma(args.b_ld)) {
                // the n tile is the same for every tile of this CTA (or pair)
                int64_t m0, n0, kb0, ke;
                int z;
                tile_of(unit0, m0, n0, z, kb0, ke);
                const uint32_t bbytes = uint32_t(nkb_full) * Lo.b_bytes * (args.b_lo ? 2u : 1u);
                if (PAIR) {
                    // each CTA's half of the B columns, counted on the leader's barrier, which
                    // expects both halves (the leader's MMAs read both)
                    const uint32_t rb = mapa_shared(smem_u32(bready), lead);
                    if (prank == 0) mbar_arrive_expect_tx(smem_u32(bready), 2u * bbytes);
                    for (int64_t kb = 0; kb < nkb_full; ++kb)
                        tma_tile<false, true>(args.tmB, args.Bm, args.b_ld, n0 + int64_t(prank) * BNS, BNS,
                                              kb0 + kb * TC_BK, bres + size_t(kb) * Lo.bres_kb, rb);
                } else {
                    mbar_arrive_expect_tx(smem_u32(bready), bbytes);
                    for (int64_t kb = 0; kb < nkb_full; ++kb) {
                        tma_tile<false>(args.tmB, args.Bm, args.b_ld, n0, BN, kb0 + kb * TC_BK,
                                        bres + size_t(kb) * Lo.bres_kb, smem_u32(bready));
                        if (args.b_lo)
                            tma_tile<false>(args.tmBlo, args.Bm, args.b_ld, n0, BN, kb0 + kb * TC_BK,
                                            bres + size_t(kb) * Lo.bres_kb + Lo.b_bytes, smem_u32(bready));
                    }
                }
            }
            bool ok = (a_dir || b_dir || a_raw || b_raw) && pair_ok;
            int64_t kbg = 0;
            int rs = 0;   // ring slot and round of kbg
            int64_t rr = 0;
            // the residual of a TMA StoreAdd epilogue: the epilogue waits on each 32 x 32 box it
            // loads, so its boxes are prefetched into L2 when the tile's operand loads start,
            // about a tile ahead of the epilogue (a streamed output: the epilogue warps prefetch
            // one chunk ahead instead, since a tile ahead the lines would not survive in L2)
            const bool pf_add = args.epi_tma && args.ep.kind == Epi::StoreAdd && !args.stream_out;
            for (int64_t t = unit0; t < ntiles && ok; t += nunits) {
                int64_t m0, n0, kb0, ke;
                int z;
                tile_of(t, m0, n0, z, kb0, ke);
                const int64_t nkb = ke > kb0 ? (ke - kb0 + TC_BK - 1) / TC_BK : 0;
                if (pf_add) {
                    for (int q = 0; q < TC_BM / 32; ++q)
                        for (int c = 0; c < BN; c += 32)
                            if (m0 + 32 * q < args.M && n0 + c < args.Nc) {
                                tma_prefetch_2d(&args.tmAdd, int(n0 + c), int(m0 + 32 * q));
                                if (args.ep.nr) tma_prefetch_2d(&args.tmNx, int(n0 + c), int(m0 + 32 * q));
                            }
                }
                for (int64_t kb = 0; kb < nkb; ++kb, ++kbg, ring_next(rs, rr, S)) {
                    const int s = rs;
                    const int64_t r = rr;
                    if (r > 0 && !mbar_wait(smem_u32(&empty[s]), uint32_t((r - 1) & 1), abort, args.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = stages + size_t(s) * Lo.stage_bytes;
                    uint8_t *sa = st, *sbb = st + Lo.a_reg;
                    const int64_t k0 = kb0 + kb * TC_BK;
                    const uint32_t txd = (a_dir ? Lo.a_bytes : 0u) + (b_dir ? Lo.b_bytes * (args.b_lo ? 2u : 1u) : 0u);
                    const uint32_t txr = (a_raw ? (args.a_mul ? 4u : 2u) * Lo.a_bytes : 0u) + (b_raw ? 2u * Lo.b_bytes : 0u);
                    if (PAIR) {
                        // bf16 A rows of this CTA and its half of the B columns, counted on the
                        // leader's barrier, which expects both CTAs' bytes
                        const uint32_t fb = mapa_shared(smem_u32(&full[s]), lead);
                        if (prank == 0) mbar_arrive_expect_tx(smem_u32(&full[s]), 2u * txd);
                        tma_tile<true, true>(args.tmA, args.A, args.a_ld, m0, TC_BM, k0, sa, fb);
                        if (!b_dir) {
                            // B resident
                        } else if (QUAD) {
                            // this CTA's half of its B half (64 rows), to itself and its counterpart
                            const int64_t row = n0 + int64_t(prank) * BNS + int64_t(pq) * (BNS / 2);
                            const uint16_t mc = uint16_t((1u << prank) | (1u << (prank + 2u)));
                            int blk = 0;
                            int64_t rr = row;
                            if (args.Bm.blk < (int64_t(1) << 30)) {
                                blk = int(row / args.Bm.blk);
                                rr = row - int64_t(blk) * args.Bm.blk;
                            }
                            // K-major: 64 rows of 128 bytes (a whole number of swizzle atoms);
                            // MN-major: one 64 x 64 box
                            const uint32_t dq = smem_u32(sbb + size_t(pq) * (size_t(BNS / 2) * 128));
                            if (args.b_ld == LD_TMA_K) tma_load_2d_quad(dq, &args.tmB[blk], int(k0), int(rr), fb, mc);
                            else tma_load_2d_quad(dq, &args.tmB[blk], int(rr), int(k0), fb, mc);
                        } else {
                            tma_tile<false, true>(args.tmB, args.Bm, args.b_ld, n0 + int64_t(prank) * BNS, BNS, k0, sbb, fb);
                        }
                    } else if (txd) {
                        const uint32_t fb = smem_u32(&full[s]);
                        mbar_arrive_expect_tx(fb, txd);
                        if (a_dir) tma_tile<true>(args.tmA, args.A, args.a_ld, m0, TC_BM, k0, sa, fb);
                        if (b_dir) {
                            tma_tile<false>(args.tmB, args.Bm, args.b_ld, n0, BN, k0, sbb, fb);
                            if (args.b_lo) tma_tile<false>(args.tmBlo, args.Bm, args.b_ld, n0, BN, k0, sbb + Lo.b_bytes, fb);
                        }
                    }
                    if (txr) {
                        const uint32_t rb = smem_u32(&rawfull[s]);
                        mbar_arrive_expect_tx(rb, txr);
                        if (a_raw) {
                            tma_tile<true>(args.tmA, args.A, args.a_ld, m0, TC_BM, k0, sa, rb);
                            if (args.a_mul) tma_tile<true>(&args.tmAmul, args.A, args.a_ld, m0, TC_BM, k0, sa + 2 * Lo.a_bytes, rb);
                        }
                        if (b_raw) tma_tile<false>(args.tmB, args.Bm, args.b_ld, n0, BN, k0, sbb, rb);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == TC_MMA_WARP) {
        // ---------------- MMA issuer
        if (lane == 0 && prank == 0 && pair_ok) {
            const bool a_mn = args.a_ld == LD_TMA_MN, b_mn = args.b_ld == LD_TMA_MN;
            const uint32_t idesc = idesc_bf16(BN, a_mn, b_mn, PAIR ? 2 * TC_BM : TC_BM);
            // a streamed raw B of 256 rows sits as two converted 128-row halves (hi, lo each):
            // one N = 128 product per half into adjacent accumulator columns
            const bool b_halves = !args.b_res && ld_raw(args.b_ld) && BN == 2 * TC_BM;
            const uint32_t idesc_h = idesc_bf16(TC_BM, a_mn, b_mn);
            bool ok = !args.b_res || mbar_wait(smem_u32(bready), 0, abort, args.status);
            if (ok) tc_fence_after();
            int64_t kbg = 0, i = 0;
            int rs = 0;   // ring slot and round of kbg
            int64_t rr = 0;
            for (int64_t t = unit0; t < ntiles && ok; t += nunits, ++i) {
                int64_t m0, n0, kb0, ke;
                int z;
                tile_of(t, m0, n0, z, kb0, ke);
                const int64_t nkb = ke > kb0 ? (ke - kb0 + TC_BK - 1) / TC_BK : 0;
                const int buf = int(i % NACC);
                const int64_t ru = i / NACC;   // earlier uses of this accumulator
                if (ru > 0 && !mbar_wait(smem_u32(&acce[buf]), uint32_t((ru - 1) & 1), abort, args.status)) break;
                tc_fence_after();
                const uint32_t dacc = tmem + uint32_t(buf * BN);
                for (int64_t kb = 0; kb < nkb; ++kb, ++kbg, ring_next(rs, rr, S)) {
                    const int s = rs;
                    const int64_t r = rr;
                    if (!mbar_wait(smem_u32(&full[s]), uint32_t(r & 1), abort, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(stages + size_t(s) * Lo.stage_bytes);
                    const uint32_t a_hi = st, a_lo = st + Lo.a_bytes;
                    uint32_t b_hi, b_lo;
                    if (args.b_res) {
                        b_hi = smem_u32(bres + size_t(kb) * Lo.bres_kb);
                        b_lo = b_hi + Lo.b_bytes;
                    } else {
                        b_hi = st + Lo.a_reg;
                        b_lo = b_hi + Lo.b_bytes;
                    }
                    const int nh = b_halves ? 2 : 1;
                    const uint32_t id = b_halves ? idesc_h : idesc;
                    for (int h = 0; h < nh; ++h) {
                        const uint32_t bh0 = b_hi + uint32_t(h) * (2 * TC_BM * 128);
                        const uint32_t bl0 = b_halves ? bh0 + TC_BM * 128 : b_lo;
                        const uint32_t dh = dacc + uint32_t(h * TC_BM);
#pragma unroll
                        for (int ks = 0; ks < TC_BK / 16; ++ks) {
                            const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
                            const uint32_t ka = a_mn ? uint32_t(ks) * 2048u : uint32_t(ks) * 32u;
                            const uint32_t kb2 = b_mn ? uint32_t(ks) * 2048u : uint32_t(ks) * 32u;
                            const uint64_t ah = a_mn ? sw128_desc_mn(a_hi + ka) : sw128_desc(a_hi + ka);
                            const uint64_t bh = b_mn ? sw128_desc_mn(bh0 + kb2) : sw128_desc(bh0 + kb2);
                            if (PAIR) mma_bf16_pair(dh, ah, bh, id, acc);
                            else mma_bf16(dh, ah, bh, id, acc);
                            if (SPLIT) {
                                const uint64_t al = a_mn ? sw128_desc_mn(a_lo + ka) : sw128_desc(a_lo + ka);
                                const uint64_t bl = b_mn ? sw128_desc_mn(bl0 + kb2) : sw128_desc(bl0 + kb2);
                                mma_bf16(dh, ah, bl, id, 1u);
                                mma_bf16(dh, al, bh, id, 1u);
                            }
                        }
                    }
                    // QUAD: the stage is released in all four CTAs (the other pair multicasts into it)
                    if (PAIR) mma_commit_pair(smem_u32(&empty[s]), QUAD ? uint16_t(0xF) : uint16_t(3u << lead));
                    else mma_commit(smem_u32(&empty[s]));
                }
                if (PAIR) mma_commit_pair(smem_u32(&accf[buf]), uint16_t(3u << lead));
                else mma_commit(smem_u32(&accf[buf]));
            }
        }
        __syncwarp();
    } else if (warp < EPIW) {
        // ---------------- epilogue (warp w: TMEM lanes 32*(w%4).., columns of half w/4)
        // A 32 x 32 chunk goes TMEM -> registers (lane = row) -> the warp's swizzled
        // shared buffer -> global.  With TMA stores (epi_tma) the fused op is applied in
        // registers, the residual of StoreAdd arrives in the buffer by TMA while TMEM is
        // read, and one lane stores the chunk; otherwise lanes store column quads.
        // ro: the residual arrives in sb and the output leaves from its own buffer ob, so the
        // next chunk's residual load is issued as soon as this chunk has read sb, and the wait
        // for the previous store to read ob is a chunk old when it is checked
        float *sb = esm + warp * (32 * 32);
        float *ob = RO ? esm + (EPIW + warp) * (32 * 32) : sb;
        const uint32_t sb_s = smem_u32(sb), ob_s = smem_u32(ob), addbar = smem_u32(&addb[warp]);
        bool ahead = false;   // ro: this warp's next chunk's residual load is in flight (lane 0)
        const int q = warp & 3, half = warp >> 2;   // lane quarter; column-chunk phase
        const int CSTEP = 32 * (EPIW / 4);
        const GemmEpilogue &ep = args.ep;
        uint32_t add_phase = 0;
        int64_t i = 0;
        // CTA pair: the accumulator is released on the leader's barrier
        const uint32_t acce_at = PAIR ? mapa_shared(smem_u32(&acce[0]), lead) : 0u;
        for (int64_t t = unit0; t < ntiles && pair_ok; t += nunits, ++i) {
            int64_t m0, n0, kb0, ke;
            int z;
            tile_of(t, m0, n0, z, kb0, ke);
            const int64_t nkb = ke > kb0 ? (ke - kb0 + TC_BK - 1) / TC_BK : 0;
            const int buf = int(i % NACC);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&accf[buf]), uint32_t((i / NACC) & 1), abort, args.status));
            tc_fence_after();
            const int64_t m0r = m0 + q * 32;
            for (int c = half * 32; c < BN; c += CSTEP) {
                const int n = int(n0) + c;
                const bool live = m0r < args.M && n < args.Nc;
                // a chunk outside the output is skipped (with TMA stores its buffer may still
                // be the source of the previous chunk's store)
                if (args.epi_tma && !live) continue;
                const bool via_tma = args.epi_tma;
                const bool add_tma = via_tma && ep.kind == Epi::StoreAdd;
                int64_t nx_m = args.M, nx_n = 0;   // this warp's next chunk (lane 0, streamed StoreAdd)
                if (via_tma) {
                    if (lane == 0) {
                        if (add_tma && args.stream_out) {
                            // L2 prefetch of this warp's next chunk: the next column chunk of the
                            // tile, else the first chunk of the CTA's next tile
                            int64_t pm = m0r, pn = int64_t(n) + CSTEP;
                            if (c + CSTEP >= BN) {
                                pm = args.M;
                                if (t + nunits < ntiles) {
                                    int64_t m1, n1, kb1, ke1;
                                    int z1;
                                    tile_of(t + nunits, m1, n1, z1, kb1, ke1);
                                    pm = m1 + q * 32;
                                    pn = n1 + half * 32;
                                }
                            }
                            if (pm < args.M && pn < args.Nc) {
                                tma_prefetch_2d(&args.tmAdd, int(pn), int(pm));
                                if (ep.nr) tma_prefetch_2d(&args.tmNx, int(pn), int(pm));
                            }
                            nx_m = pm;
                            nx_n = pn;
                        }
                        if (!RO) bulk_wait_read();   // the previous chunk's store has read the buffer
                        if (RO && ahead) {
                            ahead = false;   // the previous chunk issued this chunk's residual load
                        } else if (add_tma) {
                            const bool nxl = EXT && args.nx_tma && ep.nr != nullptr;
                            mbar_arrive_expect_tx(addbar, add_tx + (nxl ? 32 * 32 * 2 : 0));
                            if (args.stream_out) tma_load_2d_hint(sb_s, &args.tmAdd, n, int(m0r), addbar, l2_evict_first());
                            else tma_load_2d(sb_s, &args.tmAdd, n, int(m0r), addbar);
                            // the chunk's xhat rows into the bf16 buffer (free: the stores above
                            // have read it)
                            if (nxl) {
                                const uint32_t sx = smem_u32(esx + warp * (32 * 32));
                                if (args.stream_out) tma_load_2d_hint(sx, &args.tmNxl, n, int(m0r), addbar, l2_evict_first());
                                else tma_load_2d(sx, &args.tmNxl, n, int(m0r), addbar);
                            }
                        }
                    }
                    __syncwarp();
                }
                // through a normalised input: this lane's row scalars and xhat values (bf16: all 32
                // columns packed; fp32: read per quad below), issued before the TMEM load
                const bool norm = EXT && add_tma && ep.nr != nullptr;
                const bool nxt = norm && args.nx_tma;   // xhat arrives by TMA with the residual
                const int64_t nrow = m0r + lane;
                float n_mt = 0.f, n_ir = 0.f;
                uint4 n_xb[4];
                if (norm && nrow < args.M) {
                    float sdz = 0.f;
                    for (int sl = 0; sl < ep.nsl; ++sl) sdz += __ldg(ep.ndz + nrow * ep.nsl + sl);
                    n_mt = sdz * ep.inv_P;
                    n_ir = 1.f / __ldg(ep.nr + nrow);
                    if (ep.nx_bf16 && !nxt) {
                        const __nv_bfloat16 *xr = static_cast<const __nv_bfloat16 *>(ep.nx) + nrow * ep.ld + n;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
                            n_xb[g] = (n + 8 * g < args.Nc)
                                          ? (args.stream_out ? __ldcs(reinterpret_cast<const uint4 *>(xr + 8 * g))
                                                             : __ldg(reinterpret_cast<const uint4 *>(xr + 8 * g)))
                                          : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                float v[32];
                if (ok && nkb > 0) {
                    tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(buf * BN + c), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                }
                if (via_tma) {
                    int pblk = 0, pch = 0;   // ProjIn: block and first channel of the chunk
                    if (ep.kind == Epi::ProjIn) projin_col(ep, n, pblk, pch);
                    if (ep.kind == Epi::ProjIn && pblk == 0) {
                        // a = sigmoid(z + b_a) (the chunk lies within one block: N % 32 == 0)
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(ep.bias + pch + j));
                            v[j] = sigmoidf_fast(v[j] + b4.x);
                            v[j + 1] = sigmoidf_fast(v[j + 1] + b4.y);
                            v[j + 2] = sigmoidf_fast(v[j + 2] + b4.z);
                            v[j + 3] = sigmoidf_fast(v[j + 3] + b4.w);
                        }
                    }
                    bool waited = false;
                    if (nxt) {
                        mbar_wait(addbar, add_phase, abort, args.status);
                        add_phase ^= 1u;
                        waited = true;
                        const uint4 *xs = reinterpret_cast<const uint4 *>(esx + warp * (32 * 32) + lane * 32);
#pragma unroll
                        for (int g = 0; g < 4; ++g) n_xb[g] = xs[g];
                    }
                    if (norm && nrow < args.M) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            float4 x4;
                            if (ep.nx_bf16) {
                                const uint32_t w0 = (&n_xb[j >> 3].x)[(j & 7) >> 1], w1 = (&n_xb[j >> 3].x)[((j & 7) >> 1) + 1];
                                x4 = make_float4(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u),
                                                 __uint_as_float(w1 << 16), __uint_as_float(w1 & 0xFFFF0000u));
                            } else {
                                x4 = (n + j < args.Nc)
                                         ? __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(ep.nx) + nrow * ep.ld + n + j))
                                         : f4(0.f);
                            }
                            v[j] = (v[j] - x4.x * n_mt) * n_ir;
                            v[j + 1] = (v[j + 1] - x4.y * n_mt) * n_ir;
                            v[j + 2] = (v[j + 2] - x4.z * n_mt) * n_ir;
                            v[j + 3] = (v[j + 3] - x4.w * n_mt) * n_ir;
                        }
                    }
                    if (add_tma) {
                        if (!waited) {
                            mbar_wait(addbar, add_phase, abort, args.status);
                            add_phase ^= 1u;
                        }
                        if (ADD16) {
                            // this lane's row of the bf16 residual: 32 values, 64 bytes
                            uint4 rb[4];
                            const uint4 *rs = reinterpret_cast<const uint4 *>(sb) + lane * 4;
#pragma unroll
                            for (int g = 0; g < 4; ++g) rb[g] = rs[g];
                            __syncwarp();   // every row read before any lane writes its output over it
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                const uint32_t w = (&rb[j >> 3].x)[(j & 7) >> 1];
                                v[j] += __uint_as_float(w << 16);
                                v[j + 1] += __uint_as_float(w & 0xFFFF0000u);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                const float4 r4 = *reinterpret_cast<const float4 *>(sb + epi_at(lane, j >> 2));
                                v[j] += r4.x;
                                v[j + 1] += r4.y;
                                v[j + 2] += r4.z;
                                v[j + 3] += r4.w;
                            }
                        }
                    }
                    if (EXT && args.outx_tma) {
                        // the bf16 copy of this lane's row into the warp's bf16 buffer (dense 64-byte
                        // rows), stored below by TMA with the fp32 chunk: whole lines reach L2
                        uint4 *xr = reinterpret_cast<uint4 *>(esx + warp * (32 * 32) + lane * 32);
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            uint4 u;
                            u.x = pack_bf16(v[8 * g], v[8 * g + 1]);
                            u.y = pack_bf16(v[8 * g + 2], v[8 * g + 3]);
                            u.z = pack_bf16(v[8 * g + 4], v[8 * g + 5]);
                            u.w = pack_bf16(v[8 * g + 6], v[8 * g + 7]);
                            xr[g] = u;
                        }
                    } else if (EXT && ep.out_x && (ep.kind == Epi::Store || ep.kind == Epi::StoreAdd) &&
                               m0r + lane < args.M) {
                        // the bf16 copy of this lane's row: four 16-byte stores
                        __nv_bfloat16 *xr = static_cast<__nv_bfloat16 *>(ep.out_x) + (m0r + lane) * ep.ld + n;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
                            if (n + 8 * g < args.Nc) {
                                uint4 u;
                                u.x = pack_bf16(v[8 * g], v[8 * g + 1]);
                                u.y = pack_bf16(v[8 * g + 2], v[8 * g + 3]);
                                u.z = pack_bf16(v[8 * g + 4], v[8 * g + 5]);
                                u.w = pack_bf16(v[8 * g + 6], v[8 * g + 7]);
                                if (args.stream_out) __stcs(reinterpret_cast<uint4 *>(xr + 8 * g), u);
                                else *reinterpret_cast<uint4 *>(xr + 8 * g) = u;
                            }
                    }
                    if (RO) {
                        if (lane == 0) bulk_wait_read();   // the previous chunk's store has read ob
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(ob + epi_at(lane, j >> 2)) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    // orders the lanes' reads of sb and writes of ob before the bulk copies below
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (ep.kind == Epi::Partial) {
                            tma_store_3d(&args.tmO[0], n, int(m0r), z, ob_s);
                        } else if (ep.kind == Epi::ProjIn) {
                            tma_store_2d(&args.tmO[pblk], pch, int(m0r), ob_s);
                        } else if (args.stream_out) {
                            tma_store_2d_hint(&args.tmO[0], n, int(m0r), ob_s, l2_evict_first());
                        } else {
                            tma_store_2d(&args.tmO[0], n, int(m0r), ob_s);
                        }
                        if (EXT && args.outx_tma) {
                            const uint32_t sx = smem_u32(esx + warp * (32 * 32));
                            if (args.stream_out) tma_store_2d_hint(&args.tmOx, n, int(m0r), sx, l2_evict_first());
                            else tma_store_2d(&args.tmOx, n, int(m0r), sx);
                        }
                        bulk_commit();
                        if (RO && nx_m < args.M && nx_n < args.Nc) {
                            // the next chunk's residual into sb, which this chunk has read
                            mbar_arrive_expect_tx(addbar, add_tx);
                            tma_load_2d_hint(sb_s, &args.tmAdd, int(nx_n), int(nx_m), addbar, l2_evict_first());
                            ahead = true;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(sb + epi_at(lane, j >> 2)) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    __syncwarp();
                    if (m0r < args.M) epi_chunk<EXT>(args, sb, m0r, n, z, lane);
                    __syncwarp();
                }
            }
            tc_fence_before();
            if (PAIR) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acce_at + uint32_t(buf) * 8u);
            } else {
                mbar_arrive(smem_u32(&acce[buf]));
            }
            if (!ok) break;
        }
        // ro: a load issued ahead for a chunk that was not reached (an abandoned step) lands
        // before the CTA leaves
        if (lane == 0 && ahead) (void)mbar_wait(addbar, add_phase, abort, args.status);
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    // CTA pair: neither CTA leaves (or frees tensor memory) while the other may still
    // signal its barriers
    if (PAIR) cluster_sync();
    else __syncthreads();
    if (warp == TC_MMA_WARP) {
        tc_fence_after();
        if (PAIR) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
        else asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

// ---------------------------------------------------------------- launcher
static int g_num_sms = 0;
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tmap_encoder(); }

// 2-D tensor map: inner (contiguous) extent x outer extent, row pitch in bytes, box
// box_in x box_out; bf16 maps use the 128-byte swizzle of the MMA layout, fp32 (raw) maps
// none.  Out-of-range elements read as zero.
static bool make_map(CUtensorMap *m, const void *base, bool bf16, uint64_t inner, uint64_t outer,
                     uint64_t pitch_bytes, uint32_t box_in, uint32_t box_out) {
    auto enc = encode_fn();
    if (!enc || (reinterpret_cast<uintptr_t>(base) & 15u) || (pitch_bytes & 15u) || inner == 0 || outer == 0)
        return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_in, box_out};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of an fp32 epilogue output (or residual) for 32 x 32 chunks in the 128-byte
// swizzled layout of the epilogue buffer.  Rank 2, or (depth > 0) rank 3 with `depth`
// matrices `mat_stride` bytes apart (split-K partials, stored with 3-D coordinates).
static bool make_out_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t pitch_bytes,
                         uint64_t depth = 0, uint64_t mat_stride = 0) {
    auto enc = encode_fn();
    if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || (pitch_bytes & 15u) || (mat_stride & 15u) ||
        cols == 0 || rows == 0)
        return false;
    const cuuint64_t dims[3] = {cols, rows, depth > 0 ? depth : 1};
    const cuuint64_t strides[2] = {pitch_bytes, depth > 0 ? mat_stride : pitch_bytes * rows};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, depth > 0 ? 3 : 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Epilogue through TMA stores when every map builds: fp32 outputs (no bf16 copy), an
// fp32 residual, ProjIn blocks that 32-column chunks do not straddle.
// Tensor map of the bf16 output copy: 32 x 32 boxes, dense 64-byte rows in shared memory.
static bool make_outx_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t pitch_bytes) {
    auto enc = encode_fn();
    if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || (pitch_bytes & 15u) || cols == 0 || rows == 0)
        return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// add16_ok: a bf16 StoreAdd residual may arrive by TMA (pair kernels without the EXT features);
// otherwise such an epilogue stays on the lane-store path
static bool epi_maps(TcArgs &a, const GemmEpilogue &ep, int64_t M, int64_t Nc, int splits, bool add16_ok) {
    switch (ep.kind) {
    case Epi::ProjIn:
        if (ep.N % 32) return false;
        for (int b = 0; b < 3; ++b) {
            float *o = b == 0 ? ep.out0 : b == 1 ? ep.out1 : ep.out2;
            if (!make_out_map(&a.tmO[b], o, uint64_t(ep.N), uint64_t(M), uint64_t(ep.N) * 4)) return false;
        }
        return true;
    case Epi::Store:
    case Epi::StoreAdd:
        // a bf16 copy (out_x) is written by the lanes themselves, beside the TMA store
        if (!make_out_map(&a.tmO[0], ep.out0, uint64_t(Nc), uint64_t(M), uint64_t(ep.ld) * 4)) return false;
        if (ep.kind == Epi::StoreAdd) {
            const bool ok = ep.add_bf16
                                ? add16_ok && make_outx_map(&a.tmAdd, ep.add, uint64_t(Nc), uint64_t(M), uint64_t(ep.ld) * 2)
                                : make_out_map(&a.tmAdd, ep.add, uint64_t(Nc), uint64_t(M), uint64_t(ep.ld) * 4);
            if (!ok) return false;
        }
        // the normalised input is only prefetched through its map (32 x 32 boxes)
        if (ep.kind == Epi::StoreAdd && ep.nr &&
            !make_map(&a.tmNx, ep.nx, ep.nx_bf16, uint64_t(Nc), uint64_t(M), uint64_t(ep.ld) * (ep.nx_bf16 ? 2 : 4), 32, 32))
            return false;
        return true;
    case Epi::Partial:
        return make_out_map(&a.tmO[0], ep.out0, uint64_t(Nc), uint64_t(M), uint64_t(Nc) * 4, uint64_t(splits),
                            uint64_t(M) * uint64_t(Nc) * 4);
    }
    return false;
}

// Load mode an operand can use (no maps built): bf16 without a prologue product -> TMA
// straight into the MMA layout (not in split mode); fp32 without a product, 128-row tiles
// -> TMA raw + in-place conversion; otherwise register staging.
static int tma_mode(const GemmOperand &O, bool is_a, int64_t rows, int64_t K, int R, bool split3) {
    // an elementwise factor: only a k-contiguous fp32 A of one array, loaded raw
    if (O.mul && (!is_a || O.bf16 || O.s_k != 1 || O.blk < (int64_t(1) << 30) || O.s_row % 4 || R != TC_BM ||
                  (reinterpret_cast<uintptr_t>(O.mul) & 15u)))
        return LD_REG;
    const bool blocked = O.blk < (int64_t(1) << 30);
    if (blocked && (((is_a ? K : rows) + O.blk - 1) / O.blk > 3 || (is_a ? O.blk % TC_BK : O.blk % R))) return LD_REG;
    const int vec = O.bf16 ? 8 : 4;   // elements per 16 bytes
    int mode;
    if (O.s_k == 1 && O.s_row % vec == 0) mode = LD_TMA_K;
    else if (O.s_row == 1 && O.s_k % vec == 0 && R % 64 == 0) mode = LD_TMA_MN;
    else return LD_REG;
    if (O.bf16) return (split3 && !O.lo[0]) || (!split3 && O.lo[0]) ? LD_REG : mode;   // split mode: bf16 pre-split only
    // raw tiles convert 128 rows at a time: A tiles of 128 rows, B tiles of 128 or 256
    return (R == TC_BM || (!is_a && R == 2 * TC_BM)) ? (mode == LD_TMA_K ? LD_RAW_K : LD_RAW_MN) : LD_REG;
}

// Build the maps of an operand for the chosen mode; returns the mode, or LD_REG if a map
// cannot be built.
static int tma_build(CUtensorMap *maps, CUtensorMap *lo_maps, CUtensorMap *mul_map, const GemmOperand &O, int mode,
                     bool is_a, int64_t rows, int64_t K, int R) {
    if (mode == LD_REG) return LD_REG;
    const bool blocked = O.blk < (int64_t(1) << 30);
    const int nmaps = blocked ? int(((is_a ? K : rows) + O.blk - 1) / O.blk) : 1;
    const int64_t kext = (is_a && blocked) ? O.blk : K;
    const int64_t rext = (!is_a && blocked) ? O.blk : rows;
    const uint64_t es = O.bf16 ? 2 : 4;
    const bool kmaj = mode == LD_TMA_K || mode == LD_RAW_K;
    auto build = [&](CUtensorMap *m, const void *base) {
        return kmaj ? make_map(m, base, O.bf16, uint64_t(kext), uint64_t(rext), uint64_t(O.s_row) * es, 64, uint32_t(R))
                    : make_map(m, base, O.bf16, uint64_t(rext), uint64_t(kext), uint64_t(O.s_k) * es, 64, 64);
    };
    for (int i = 0; i < nmaps; ++i) {
        if (!build(&maps[i], O.p[i])) return LD_REG;
        if (O.lo[0] && (!lo_maps || !build(&lo_maps[i], O.lo[i]))) return LD_REG;
    }
    if (O.mul && (!mul_map || !build(mul_map, O.mul))) return LD_REG;
    return mode;
}

template <bool ABF, bool BBF, bool SPLIT, bool REGS = true, bool EXT = true>
static cudaError_t launch_tc_t(const TcArgs &a, unsigned grid, size_t smem, cudaStream_t st) {
    auto kern = k_gemm_tc<ABF, BBF, SPLIT, REGS, false, EXT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, TC_THREADS_P, smem, st>>>(a);
    return cudaGetLastError();
}

// The CTA-pair instantiation (bf16 operands, all by TMA): launched as clusters of two, or
// of four (two pairs sharing B by multicast).
using PairKernel = void (*)(TcArgs);
static PairKernel pair_kernel(bool ext = false, bool quad = false) {
    if (quad)
        return ext ? k_gemm_tc<false, false, false, false, true, true, true>
                   : k_gemm_tc<false, false, false, false, true, false, true>;
    return ext ? k_gemm_tc<false, false, false, false, true, true> : k_gemm_tc<false, false, false, false, true, false>;
}
static cudaLaunchConfig_t pair_config(unsigned grid, size_t smem, cudaStream_t st, cudaLaunchAttribute *attr,
                                      unsigned cluster = 2) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(TC_THREADS_P, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}
// Clusters of two (pairs) or four (quads) CTAs that can be resident at once with this much
// shared memory (0 if none).
static int pair_slots(size_t smem, bool quad = false) {
    static size_t cached_smem[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    static int cached[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
    static bool cached_quad[8] = {false, false, false, false, false, false, false, false};
    static int next = 0;
    for (int i = 0; i < 8; ++i)
        if (cached[i] >= 0 && cached_smem[i] == smem && cached_quad[i] == quad) return cached[i];
    if (cudaFuncSetAttribute(pair_kernel(false, quad), cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
        return 0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config(quad ? 4 : 2, smem, nullptr, attr, quad ? 4 : 2);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, pair_kernel(false, quad), &cfg) != cudaSuccess) n = 0;
    cached_smem[next] = smem;
    cached[next] = n;
    cached_quad[next] = quad;
    next = (next + 1) % 8;
    return n;
}
static cudaError_t launch_pair(const TcArgs &a, unsigned grid, size_t smem, cudaStream_t st, bool ext,
                               bool quad = false) {
    cudaError_t e =
        cudaFuncSetAttribute(pair_kernel(ext, quad), cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config(grid, smem, st, attr, quad ? 4 : 2);
    return cudaLaunchKernelEx(&cfg, pair_kernel(ext, quad), a);
}

// Whether a streamed StoreAdd pair product with a short K keeps B resident and gives its
// epilogue warps separate residual and output buffers (TC_RO_*).
static int g_ro_mode = -1;
static bool ro_enabled() {
    if (g_ro_mode < 0) {
        const char *v = getenv("ADJ_GEMM_RO");
        g_ro_mode = (v && v[0] == '0') ? 0 : 1;
    }
    return g_ro_mode == 1;
}

// Whether pair GEMMs with a long K (a mainloop bound by operand delivery) run as quads.
static int g_quad_mode = -1;
static bool quad_enabled() {
    if (g_quad_mode < 0) {
        const char *v = getenv("ADJ_GEMM_QUAD");
        g_quad_mode = (v && v[0] == '0') ? 0 : 1;
    }
    return g_quad_mode == 1;
}

// Whether GEMMs whose operands are both bf16 and both loaded by TMA run as CTA pairs.
static int g_pair_mode = -1;   // -1: not read yet
static bool pair_enabled() {
    if (g_pair_mode < 0) {
        const char *v = getenv("ADJ_GEMM_PAIR");
        g_pair_mode = (v && v[0] == '0') ? 0 : 1;
    }
    return g_pair_mode == 1;
}

cudaError_t launch_gemm_tc(int64_t M, int64_t Nc, int64_t K, const GemmOperand &A, const GemmOperand &Bm,
                           const GemmEpilogue &ep, int splits, bool split3, unsigned *status, cudaStream_t st,
                           int *splits_used, bool *csum_done) {
    if (csum_done) *csum_done = false;
    if (M <= 0 || Nc <= 0) return cudaSuccess;
    if (splits < 1) splits = 1;
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    TcArgs a;
    memset(&a, 0, sizeof(a));
    a.M = M; a.Nc = Nc; a.K = K; a.splits = splits;
    int64_t kper = (K + splits - 1) / splits;
    a.kper = (kper + TC_BK - 1) / TC_BK * TC_BK;
    // Tile width: the widest (<= 256, a multiple of 32) whose stages fit; B resident when its
    // whole k extent fits next to two A stages and the epilogue buffer.  A streamed fp32 B
    // that TMA can load raw takes 128-column tiles (the in-place conversion works on 128 rows).
    const size_t budget = 227 * 1024 - 1024 - TC_EPI_SMEM - 512;
    const int a_mode = tma_mode(A, true, M, K, TC_BM, split3);
    const bool a_mul = A.mul && ld_raw(a_mode);
    int BN = int(Nc < 256 ? (Nc + 31) / 32 * 32 : 256);
    int S = 0, b_mode = LD_REG;
    // bf16 operands that TMA loads straight into the MMA layout run as CTA pairs (below),
    // with six streamed stages: no resident B, whose two stages leave too few operand bytes
    // in flight per SM to cover the HBM latency of a short-K product
    const bool pair_cand = pair_enabled() && !split3 && !a_mul && A.bf16 && Bm.bf16 && !A.lo[0] && !Bm.lo[0] &&
                           (a_mode == LD_TMA_K || a_mode == LD_TMA_MN) && BN % TC_BM == 0;
    for (int next = BN;; BN = next) {
        if (BN == 0) return cudaErrorInvalidConfiguration;
        next = BN > 32 ? (BN / 2 + 31) / 32 * 32 : 0;
        const TcLayout res = tc_layout(BN, a.kper, true, split3, ld_raw(a_mode), false, a_mul);
        a.b_res = splits == 1 && size_t(res.bres_bytes) + 2 * size_t(res.stage_bytes) <= budget;
        if (pair_cand && BN % TC_BM == 0) {
            const int bm = tma_mode(Bm, false, Nc, K, BN, split3);
            if (bm == LD_TMA_K || bm == LD_TMA_MN) a.b_res = false;
        }
        b_mode = tma_mode(Bm, false, Nc, K, BN, split3);
        if (a.b_res && ld_raw(b_mode)) b_mode = LD_REG;          // a resident B is converted once, by registers
        if (!a.b_res && !Bm.bf16 && !Bm.mul && BN > TC_BM && BN != 2 * TC_BM &&
            tma_mode(Bm, false, Nc, K, TC_BM, split3) != LD_REG) {
            next = TC_BM;                                         // take 128-column tiles to load B raw
            continue;
        }
        const TcLayout Lt = tc_layout(BN, a.kper, a.b_res, split3, ld_raw(a_mode), ld_raw(b_mode), a_mul);
        S = int((budget - Lt.bres_bytes) / Lt.stage_bytes);
        if (S >= 2) break;
    }
    if (S > 6) S = 6;
    // CTA pairs: both operands bf16 by TMA (no conversion, no resident B), tiles of 256
    // rows x BN with BN / 2 columns of B staged in each CTA
    bool pair = pair_cand && !a.b_res && (b_mode == LD_TMA_K || b_mode == LD_TMA_MN) && BN % TC_BM == 0;
    int slots = 0;
    // pairs with many tiles each (no split) and a short K use 16 epilogue warps, with one
    // stage fewer; a long K keeps the stage (its mainloop outlasts the epilogue of 8 warps)
    int epiw = (pair && splits == 1 && K <= 1024) ? TC_MAX_EPI_WARPS : TC_EPI_WARPS;
    // a pair epilogue with a bf16 output copy stages it per warp (2 KB) and stores it by TMA
    const bool outx = pair_cand && ep.out_x != nullptr && (ep.kind == Epi::Store || ep.kind == Epi::StoreAdd);
    const size_t epi_bytes = size_t(epiw) * TC_CHUNK_BYTES * (outx ? 3 : 2) / 2;
    const size_t bar_bytes = size_t(3 * 6 + 6 + TC_MAX_EPI_WARPS) * 8;
    if (pair) {
        const TcLayout Lp = tc_layout(BN / 2, a.kper, false, false, false, false, false);
        const size_t budget_p = 227 * 1024 - 1024 - epi_bytes - bar_bytes;
        int Sp = int(budget_p / Lp.stage_bytes);
        if (Sp > 6) Sp = 6;
        const size_t smem_p = 1024 + size_t(Sp) * Lp.stage_bytes + epi_bytes + bar_bytes;
        slots = Sp >= 2 ? pair_slots(smem_p) : 0;
        if (slots > 0) S = Sp;
        else pair = false;
    }
    // quads: two pairs on neighbouring 256-row tiles share B by multicast, for a long K (a
    // mainloop bound by operand delivery) and B spread over several n tiles (a single n tile
    // of B stays close in L2 anyway); at least two pair rows of tiles, whole 64-row halves
    bool quad = false;
    if (pair && quad_enabled() && K > 1024 && (Nc + BN - 1) / BN >= 2 && (M + 2 * TC_BM - 1) / (2 * TC_BM) >= 2 &&
        (BN / 2) % 64 == 0) {
        const TcLayout Lp = tc_layout(BN / 2, a.kper, false, false, false, false, false);
        const size_t smem_p = 1024 + size_t(S) * Lp.stage_bytes + epi_bytes + bar_bytes;
        const int q = pair_slots(smem_p, true);
        if (q > 0) {
            quad = true;
            slots = q;
        }
    }
    // a streamed StoreAdd pair product whose B half fits resident (the output projection):
    // resident B, TC_RO_STAGES A stages, TC_RO_EPI_WARPS epilogue warps with a residual and an
    // output buffer each; every pair then keeps one n tile, so the pairs are a multiple of the
    // n tiles
    const bool ext = ep.nr != nullptr || ep.out_x != nullptr;   // the EXT epilogue features
    bool ro = false;
    if (pair && !quad && ro_enabled() && splits == 1 && ep.kind == Epi::StoreAdd && !ext &&
        uint64_t(M) * uint64_t(Nc) * 4u > (uint64_t(256) << 20) && epi_maps(a, ep, M, Nc, splits, true)) {
        const TcLayout Lr = tc_layout(BN / 2, a.kper, TC_RO_BRES, false, false, false, false);
        const size_t smem_r = 1024 + size_t(Lr.bres_bytes) + size_t(TC_RO_STAGES) * Lr.stage_bytes +
                              size_t(TC_RO_EPI_WARPS) * TC_CHUNK_BYTES * 2 + bar_bytes;
        const int nt = TC_RO_BRES ? int((Nc + BN - 1) / BN) : 1;
        const int q = smem_r <= size_t(227) * 1024 ? pair_slots(smem_r) : 0;
        if (q >= nt) {
            ro = true;
            a.b_res = TC_RO_BRES;
            S = TC_RO_STAGES;
            epiw = TC_RO_EPI_WARPS;
            slots = q / nt * nt;
        }
    }
    const int64_t rows_per_tile = quad ? 4 * TC_BM : pair ? 2 * TC_BM : TC_BM;
    const int64_t units = pair ? slots : g_num_sms;   // tiles in flight: clusters (pairs, quads) or CTAs
    // split K no further than one wave of CTAs: every CTA then owns exactly one tile
    {
        const int64_t per_split = ((Nc + BN - 1) / BN) * ((M + rows_per_tile - 1) / rows_per_tile);
        const int64_t cap = (units / ((Nc + BN - 1) / BN)) * ((Nc + BN - 1) / BN);
        if (splits > 1 && int64_t(splits) * per_split > cap) {
            splits = int(cap / per_split > 1 ? cap / per_split : 1);
            a.splits = splits;
            kper = (K + splits - 1) / splits;
            a.kper = (kper + TC_BK - 1) / TC_BK * TC_BK;
        }
    }
    if (splits_used) *splits_used = splits;
    a.BN = BN;
    a.stages = S;
    a.nacc = 2;   // the epilogue of one tile overlaps the mainloop of the next
    a.epiw = pair ? epiw : TC_EPI_WARPS;
    a.n_tiles = int((Nc + BN - 1) / BN);
    a.m_tiles = int((M + rows_per_tile - 1) / rows_per_tile);
    a.A = A; a.Bm = Bm; a.ep = ep; a.status = status;
    a.a_ld = tma_build(a.tmA, nullptr, &a.tmAmul, A, a_mode, true, M, K, TC_BM);
    a.b_ld = tma_build(a.tmB, a.tmBlo, nullptr, Bm, b_mode, false, Nc, K, quad ? BN / 4 : pair ? BN / 2 : BN);
    if (pair && (a.a_ld != a_mode || a.b_ld != b_mode)) return cudaErrorInvalidValue;   // a map did not build
    a.a_mul = a_mul && a.a_ld != LD_REG;
    a.epi_tma = epi_maps(a, ep, M, Nc, splits, pair && !ext);
    a.add16 = a.epi_tma && ep.kind == Epi::StoreAdd && ep.add_bf16;
    a.outx_tma = outx && pair && a.epi_tma &&
                 make_outx_map(&a.tmOx, ep.out_x, uint64_t(Nc), uint64_t(M), uint64_t(ep.ld) * 2);
    a.nx_tma = a.outx_tma && ep.kind == Epi::StoreAdd && ep.nr && ep.nx_bf16 &&
               make_outx_map(&a.tmNxl, ep.nx, uint64_t(Nc), uint64_t(M), uint64_t(ep.ld) * 2);
    // a residual stream far larger than L2 (129 MB): its output lines cannot serve a later
    // reader from L2, so they go out first
    a.stream_out = a.epi_tma && ep.kind == Epi::StoreAdd && uint64_t(M) * uint64_t(Nc) * 4u > (uint64_t(256) << 20);
    a.ro = ro && a.stream_out;
    if (ro && !a.ro) return cudaErrorInvalidValue;   // its maps were built above
    a.b_lo = Bm.lo[0] && a.b_ld != LD_REG;
    // the layout was sized for the modes asked for; a mode that fell back to registers
    // uses only part of its region
    const TcLayout L = tc_layout(pair ? BN / 2 : BN, a.kper, a.b_res, split3, ld_raw(a_mode), ld_raw(b_mode), a_mul);
    const size_t smem = 1024 + size_t(L.bres_bytes) + size_t(S) * L.stage_bytes +
                        size_t(a.epiw) * TC_CHUNK_BYTES * ((pair && outx) ? 3 : 2) / 2 +
                        (a.ro ? size_t(a.epiw) * TC_CHUNK_BYTES : 0) + bar_bytes;
    const int64_t ntiles = int64_t(a.n_tiles) * a.m_tiles * splits;
    if (pair) {
        a.ep.csum = nullptr;
        if (csum_done) *csum_done = false;
        const int64_t nclus = ntiles < slots ? ntiles : slots;
        return launch_pair(a, unsigned((quad ? 4 : 2) * nclus), smem, st, ext, quad);
    }
    int64_t grid = ntiles;
    if (grid > g_num_sms) grid = (g_num_sms / a.n_tiles) * a.n_tiles;
    if (grid < a.n_tiles) grid = a.n_tiles;
    if (grid > ntiles) grid = ntiles;
    // the fused column sums need a raw row-contiguous B, streamed, and one tile per CTA
    const bool csum = ep.csum && ep.kind == Epi::Partial && a.b_ld == LD_RAW_MN && !a.b_res && grid == ntiles &&
                      ep.csum_n > 0 && ep.csum_n <= Nc;
    if (!csum) a.ep.csum = nullptr;
    if (csum_done) *csum_done = csum;
    const bool need_regs = a.a_ld == LD_REG || (!a.b_res && a.b_ld == LD_REG) || (a.b_res && !ld_tma(a.b_ld));
    if (!need_regs) {
        if (split3) {
            if (ext) return launch_tc_t<false, false, true, false, true>(a, unsigned(grid), smem, st);
            return launch_tc_t<false, false, true, false, false>(a, unsigned(grid), smem, st);
        }
        if (ext) return launch_tc_t<false, false, false, false, true>(a, unsigned(grid), smem, st);
        return launch_tc_t<false, false, false, false, false>(a, unsigned(grid), smem, st);
    }
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
