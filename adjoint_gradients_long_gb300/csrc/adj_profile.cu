// adj_profile.cu -- launch counting and per-kernel CUDA-event timing of libadj.so.
// Every launcher runs inside a ProfScope; when profiling is on, the scope records a
// CUDA event before and after the launch on the launching stream, and
// adj_profile_read() sums the elapsed times per kernel kind.
#include <atomic>
#include <mutex>
#include <vector>

#include "adj_internal.cuh"
#include "adj_profile.cuh"

namespace adj {

namespace {
struct Rec {
    cudaEvent_t a, b;
};
std::mutex g_mu;
std::atomic<bool> g_on{false};
std::atomic<unsigned long long> g_launches{0};
std::vector<Rec> g_recs[K_COUNT];
std::vector<cudaEvent_t> g_pool;

const char *g_names[K_COUNT] = {"proj_in", "fwd_scan", "proj_out", "loss", "cot_proj", "win_scan",
                                "bwd_scan", "param_dW_in", "param_dW_o", "param_reduce", "colsum",
                                "input_grad", "rms_norm", "rms_norm_bwd", "weight_prep",
                                "sel_proj", "sel_fwd", "sel_bwd", "sel_dW", "sel_dx"};

cudaEvent_t take() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

ProfScope::ProfScope(KernelId id, cudaStream_t st, int launches) : id_(id), st_(st), on_(g_on.load()) {
    g_launches.fetch_add(launches);
    if (on_) {
        std::lock_guard<std::mutex> lk(g_mu);
        a_ = take();
        b_ = take();
        cudaEventRecord(a_, st_);
    }
}

ProfScope::~ProfScope() {
    if (on_) {
        cudaEventRecord(b_, st_);
        std::lock_guard<std::mutex> lk(g_mu);
        g_recs[id_].push_back(Rec{a_, b_});
    }
}

}  // namespace adj

using namespace adj;

extern "C" {

void adj_profile_enable(int on) { g_on.store(on != 0); }

void adj_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto &v : g_recs) {
        for (auto &r : v) {
            g_pool.push_back(r.a);
            g_pool.push_back(r.b);
        }
        v.clear();
    }
}

int adj_profile_kernels(void) { return K_COUNT; }

const char *adj_profile_name(int id) { return (id >= 0 && id < K_COUNT) ? g_names[id] : nullptr; }

adj_status adj_profile_read(int id, int64_t *launches, double *total_ms) {
    if (id < 0 || id >= K_COUNT || !launches || !total_ms) return ADJ_EINVAL;
    std::lock_guard<std::mutex> lk(g_mu);
    double ms = 0.0;
    for (auto &r : g_recs[id]) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return ADJ_ECUDA;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return ADJ_ECUDA;
        ms += t;
    }
    *launches = int64_t(g_recs[id].size());
    *total_ms = ms;
    return ADJ_OK;
}

unsigned long long adj_launch_count(void) { return g_launches.load(); }

}  // extern "C"
