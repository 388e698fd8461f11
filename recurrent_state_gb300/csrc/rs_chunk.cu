// rs_chunk.cu -- the chunk-parallel prefill (rs_chunk.cuh) on the FP32 state
// layout: instantiations and launch (dk = dv = 128).
#include "rs_chunk.cuh"

namespace rs {

namespace {

template <bool KDA>
cudaError_t by_types(const StepLaunch &L, PrefillParams &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32) return run<KDA, false, false, false, __nv_bfloat16, float>(P, s);
    if (L.in_dt == RS_BF16 && L.out_dt == RS_BF16) return run<KDA, false, false, false, __nv_bfloat16, __nv_bfloat16>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<KDA, false, false, false, float, float>(P, s);
    if (L.in_dt == RS_F16 && L.out_dt == RS_F32) return run<KDA, false, false, false, __half, float>(P, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_prefill_chunked(const StepLaunch &L, PrefillParams &P, cudaStream_t s) {
    if (L.D != 128) return cudaErrorNotSupported;
    if (L.khi >= 0) return launch_prefill_chunked_mixed(L, P, s);
    return L.kda ? by_types<true>(L, P, s) : by_types<false>(L, P, s);
}

}  // namespace rs
