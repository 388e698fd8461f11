// rs_chunk_damp.cu -- the chunk-parallel prefill (rs_chunk.cuh) on the
// DAMP-exact layout (16 FP16 rows, INT8 scales per group of 32 columns, value
// scaling; dk = dv = 128): instantiations and launch, both requantisation
// arithmetics.
#include "rs_chunk.cuh"

namespace rs {

namespace {

template <bool KDA, bool FUSED>
cudaError_t by_types(const StepLaunch &L, PrefillParamsDamp &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32) return run<KDA, true, true, FUSED, __nv_bfloat16, float>(P, s);
    if (L.in_dt == RS_BF16 && L.out_dt == RS_BF16) return run<KDA, true, true, FUSED, __nv_bfloat16, __nv_bfloat16>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<KDA, true, true, FUSED, float, float>(P, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_prefill_chunked_damp(const StepLaunch &L, PrefillParamsDamp &P, cudaStream_t s) {
    if (L.D != 128 || L.khi != KHM) return cudaErrorNotSupported;
    if (L.fused) return L.kda ? by_types<true, true>(L, P, s) : by_types<false, true>(L, P, s);
    return L.kda ? by_types<true, false>(L, P, s) : by_types<false, false>(L, P, s);
}

}  // namespace rs
