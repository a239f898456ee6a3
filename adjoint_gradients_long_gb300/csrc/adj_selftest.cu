// adj_selftest.cu -- adj_selftest_waits: exercises the bounded device waits the kernels
// use (a look-back flag and an mbarrier) on objects that are never released, so the
// give-up path runs: the waits time out, record ADJ_ETIMEOUT in the workspace status
// word and the kernel returns.  Nothing faults or hangs; the context stays usable.
#include "adj_internal.cuh"
#include "adj_ptx.cuh"

namespace {

__global__ void k_selftest_waits(unsigned *status, unsigned *flag, int which) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x != 0) return;
    if (which & 1) {
        // the look-back flag wait: *flag stays 0
        (void)adj::wait_flag(flag, status);
    }
    if (which & 2) {
        // an mbarrier expecting one arrival that never comes
        abort = 0;
        const uint32_t b = adj::smem_u32(&bar);
        adj::mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        (void)adj::mbar_wait(b, 0, &abort, status);
    }
}

}  // namespace

extern "C" adj_status adj_selftest_waits(void *ws, size_t ws_bytes, int which, void *stream) {
    if (!ws) return ADJ_EINVAL;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return ADJ_EALIGN;
    if (ws_bytes < adj::WS_HEADER + 256) return ADJ_EWORKSPACE;
    if (which < 1 || which > 3) return ADJ_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned *flag = reinterpret_cast<unsigned *>(static_cast<char *>(ws) + adj::WS_HEADER);
    if (cudaMemsetAsync(flag, 0, 256, st) != cudaSuccess) return ADJ_ECUDA;
    k_selftest_waits<<<1, 32, 0, st>>>(static_cast<unsigned *>(ws), flag, which);
    return cudaGetLastError() == cudaSuccess ? ADJ_OK : ADJ_ECUDA;
}
