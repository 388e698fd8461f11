// rs_prefill_mixed.cu -- prefill chunks on the mixed FP16/INT8 layout
// (dk = 128, 16 FP16 rows), both requantisation modes (the kernel:
// rs_prefill.cuh).
#include "rs_prefill.cuh"

namespace rs {

cudaError_t launch_prefill_mixed(const StepLaunch &L, PrefillParams &P, cudaStream_t s) {
    return by_mode<false>(L, P, s);
}

}  // namespace rs
