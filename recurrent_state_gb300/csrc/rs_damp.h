// rs_damp.h -- launch interface of the DAMP-exact storage kernels: INT8 rows
// in groups of 32 values along dv with one FP32 scale per group, and value
// scaling (DAMP Appendix A.1, A.3 Eq. 17-18, A.4).  Internal to the library.
#pragma once

#include "rs_internal.h"

namespace rs {

constexpr int kDampGroup = 32;           // values per INT8 scale group
constexpr int kMaxValueScales = 4096;    // Hv * dv value-scaling factors carried in the launch params

// Step parameters plus the value-scaling factors c' [Hv][dv] (launch params:
// the library allocates no device memory for them).
struct StepParamsDamp : StepParamsPi {
    float cs[kMaxValueScales];
};

struct ConvertParamsDamp : ConvertParamsPi {
    float cs[kMaxValueScales];
};

struct PrefillParamsDamp : PrefillParams {
    float cs[kMaxValueScales];
};

cudaError_t launch_step_damp_decode(const StepLaunch &L, StepParamsDamp &P, cudaStream_t s);
cudaError_t launch_prefill_damp(const StepLaunch &L, PrefillParamsDamp &P, cudaStream_t s);
// rs_chunk_damp.cu: the chunk-parallel prefill on the tensor cores, DAMP-exact tiles (groups of 32)
cudaError_t launch_prefill_chunked_damp(const StepLaunch &L, PrefillParamsDamp &P, cudaStream_t s);
cudaError_t launch_convert_damp(int D, int khi, ConvertParamsDamp &P, cudaStream_t s);

}  // namespace rs
