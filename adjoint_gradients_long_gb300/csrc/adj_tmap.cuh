// adj_tmap.cuh -- host-side construction of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so the library needs no -lcuda).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace adj {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Rank-2 fp32 map over a row-major [rows, cols] array with the given row pitch, box
// box_cols x box_rows, no swizzle; elements outside the array read as zero.
inline bool tmap_rows_f32(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t pitch_bytes,
                          uint32_t box_cols, uint32_t box_rows) {
    auto enc = tmap_encoder();
    if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || (pitch_bytes & 15u) || cols == 0 || rows == 0)
        return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace adj
