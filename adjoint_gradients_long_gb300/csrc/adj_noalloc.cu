// adj_noalloc.cu -- adj_fwd_scan_noalloc: the forward pass of one layer for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running where another component owns all
// device memory (a host application with its own pool), callbacks that must not
// allocate, or plugins loaded into a process whose allocator they may not touch.  For
// them this entry point takes its scratch from a file-scope device array instead of a
// caller workspace.  The array is part of the library image: every GPU that loads the
// library holds NOALLOC_SCRATCH_BYTES of it until the process exits.
//
// Host code cannot use the array's name as a device address (in host code it names a
// host-side stand-in).  The first call on each device, with that device current, asks
// the runtime for the array's device address (cudaGetSymbolAddress) and caches it; make
// that first call before any stream capture.  Every call shares the one array and it
// keeps the last call's contents, so calls that overlap on the GPU (different streams,
// or different host threads without ordering) race.  The calls this entry point makes
// are the same kernels adj_fwd_scan launches, plus cudaMemsetAsync / cudaMemcpyAsync on
// the array; it calls no cudaMalloc, cudaFree or other allocating routine.
#include <mutex>

#include "adj_internal.cuh"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(32) << 20;   // 32 MiB per device
constexpr int MAX_DEVICES = 128;

__device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_addr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device (set up once per device).
adj_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return ADJ_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ADJ_ECUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return ADJ_OK;
}

}  // namespace

extern "C" adj_status adj_fwd_scan_noalloc(const adj_dims *dims, const adj_weights *w, const void *xhat,
                                           const float *xres, float *a, float *c, float *h, float *y, void *y_x,
                                           unsigned *status, void *stream) {
    const size_t need = adj_workspace_bytes(dims, ADJ_OP_FWD, 0);
    if (need == 0) return dims ? ADJ_ESHAPE : ADJ_EINVAL;
    if (need > NOALLOC_SCRATCH_BYTES) return ADJ_EWORKSPACE;   // too large for the static scratch
    if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return ADJ_EALIGN;
    void *ws = nullptr;
    adj_status s = scratch_address(&ws);
    if (s != ADJ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // adj_fwd_scan validates every argument before it launches anything: any status but
    // ADJ_OK and ADJ_ECUDA means nothing was launched and the array is untouched.
    s = adj_fwd_scan(dims, w, xhat, xres, a, c, h, y, y_x, ws, NOALLOC_SCRATCH_BYTES, stream);
    if (s != ADJ_OK && s != ADJ_ECUDA) return s;
    // Kernels may have run (ADJ_ECUDA can come after some launches): report the device
    // status word, then clear the header, so that the next call starts from a zero
    // status word whatever happened here.  The look-back descriptors are reset by the
    // scan launcher itself.
    adj_status out = s;
    if (status && cudaMemcpyAsync(status, ws, sizeof(unsigned), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        out = ADJ_ECUDA;
    if (cudaMemsetAsync(ws, 0, adj::WS_HEADER, st) != cudaSuccess) out = ADJ_ECUDA;
    return out;
}
