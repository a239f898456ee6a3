// adj_selftest.cu -- adj_selftest_waits: runs the bounded device waits of the kernels on
// objects that are never released, so their give-up path runs: the waits time out,
// record ADJ_ETIMEOUT in the workspace status word and the kernels return.  Nothing
// faults or hangs; the context stays usable.
//   which & 1: the scans' decoupled look-back.  The forward state scan (the product
//              kernel, unchanged) runs over a small problem whose first chunk is never
//              launched, so every other chunk waits for a predecessor that never
//              publishes, until the look-back's round limit.
//   which & 2: the mbarrier wait of TMA staging and the GEMM pipeline, on a barrier
//              that expects one arrival that never comes.
#include "adj_internal.cuh"
#include "adj_ptx.cuh"

namespace {

constexpr int ST_T = 8 * 96, ST_N = 128;   // eight forward-scan chunks of one 128-channel slice

__global__ void k_selftest_mbar(unsigned *status) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x != 0) return;
    abort = 0;
    const uint32_t b = adj::smem_u32(&bar);
    adj::mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    (void)adj::mbar_wait(b, 0, &abort, status);
}

size_t arr_bytes() { return size_t(ST_T) * ST_N * sizeof(float); }

}  // namespace

extern "C" size_t adj_selftest_ws_bytes(void) {
    return adj::WS_HEADER + 3 * arr_bytes() + ((adj::scan_ws_bytes(1, ST_T, ST_N) + 255) & ~size_t(255));
}

extern "C" adj_status adj_selftest_waits(void *ws, size_t ws_bytes, int which, void *stream) {
    if (!ws) return ADJ_EINVAL;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return ADJ_EALIGN;
    if (ws_bytes < adj_selftest_ws_bytes()) return ADJ_EWORKSPACE;
    if (which < 1 || which > 3) return ADJ_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned *status = static_cast<unsigned *>(ws);
    if (which & 1) {
        char *p = static_cast<char *>(ws) + adj::WS_HEADER;
        float *a = reinterpret_cast<float *>(p), *u = a + size_t(ST_T) * ST_N, *h = u + size_t(ST_T) * ST_N;
        void *scan = p + 3 * arr_bytes();
        if (cudaMemsetAsync(a, 0, 2 * arr_bytes(), st) != cudaSuccess) return ADJ_ECUDA;
        if (adj::launch_fwd_scan(a, u, h, 1, ST_T, ST_N, scan, status, st, /*withhold_first=*/true) != cudaSuccess)
            return ADJ_ECUDA;
    }
    if (which & 2) {
        k_selftest_mbar<<<1, 32, 0, st>>>(status);
        if (cudaGetLastError() != cudaSuccess) return ADJ_ECUDA;
    }
    return ADJ_OK;
}
