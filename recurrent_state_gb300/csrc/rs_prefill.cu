// rs_prefill.cu -- prefill chunks, FP32 layout, and the entry point that
// dispatches by layout (the kernel: rs_prefill.cuh).
#include "rs_prefill.cuh"

namespace rs {

cudaError_t launch_prefill(const StepLaunch &L, PrefillParams &P, cudaStream_t s) {
    if (L.D != 128) return cudaErrorNotSupported;
    if (L.khi < 0)
        return L.kda ? by_types<128, -1, true, false, false>(L, P, s) : by_types<128, -1, false, false, false>(L, P, s);
    if (L.khi != 16) return cudaErrorNotSupported;
    return launch_prefill_mixed(L, P, s);
}

}  // namespace rs
