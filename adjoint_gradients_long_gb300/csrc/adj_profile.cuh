// adj_profile.cuh -- kernel kinds and the launch scope used by the profiler.
#pragma once
#include <cuda_runtime.h>

namespace adj {

enum KernelId {
    K_PROJ_IN = 0,
    K_FWD_SCAN,
    K_PROJ_OUT,
    K_LOSS,
    K_COT_PROJ,
    K_WIN_SCAN,
    K_BWD_SCAN,
    K_PARAM_DWIN,
    K_PARAM_DWO,
    K_PARAM_REDUCE,
    K_COLSUM,
    K_INPUT_GRAD,
    K_RMS_NORM,
    K_RMS_NORM_BWD,
    K_WEIGHT_PREP,
    K_SEL_PROJ,
    K_SEL_FWD,
    K_SEL_BWD,
    K_SEL_DW,
    K_SEL_DX,
    K_COUNT
};

// Counts `launches` kernel launches and, while profiling is on, brackets them with
// CUDA events on `st`.
class ProfScope {
  public:
    ProfScope(KernelId id, cudaStream_t st, int launches = 1);
    ~ProfScope();
    ProfScope(const ProfScope &) = delete;
    ProfScope &operator=(const ProfScope &) = delete;

  private:
    KernelId id_;
    cudaStream_t st_;
    bool on_;
    cudaEvent_t a_ = nullptr, b_ = nullptr;
};

}  // namespace adj
