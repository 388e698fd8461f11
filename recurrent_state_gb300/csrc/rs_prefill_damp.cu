// rs_prefill_damp.cu -- prefill chunks and multi-token replay on the
// DAMP-exact layout (INT8 groups of 32, value scaling), both requantisation
// modes (the kernel: rs_prefill.cuh).
#include "rs_prefill.cuh"

namespace rs {

cudaError_t launch_prefill_damp(const StepLaunch &L, PrefillParamsDamp &P, cudaStream_t s) {
    if (L.D != 128 || L.khi != 16) return cudaErrorNotSupported;
    return by_mode<true>(L, P, s);
}

}  // namespace rs
