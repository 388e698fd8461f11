// rs_step_mixed_replay.cu -- instantiations of the step kernel for the mixed
// FP16/INT8 layout (dk = dv = 128, 16 FP16 rows per head), speculative replay of up to 8 tokens.
#include "rs_step.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

template <int D, int KHI, bool KDA, int MAXT, typename TI, typename TO, bool FUSED>
cudaError_t run(StepParamsPi &P, cudaStream_t s) {
    using Sh = StepShape<D, KHI, KDA, TI>;
    auto kern = step_kernel<D, KHI, KDA, MAXT, TI, TO, StepParamsPi, FUSED>;
    const int region = Sh::region_bytes(P.T_max);
    const int header = 128 + (P.Hv * D + 127) / 128 * 128;
    const int smax = device_max_smem_optin();
    int G = step_threads(MAXT) / D;
    while (G > 1 && header + G * region > smax) --G;
    if (header + G * region > smax) return cudaErrorNotSupported;
    const int groups_needed = (P.B * P.Hv + G - 1) / G;
    int grid = device_sm_count();
    if (grid > groups_needed) grid = groups_needed;
    if (grid < 1) grid = 1;
    P.header_bytes = header;
    P.region_bytes = region;
    const int smem = header + G * region;
    cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(G * D), smem, s, P);
}

template <bool KDA, bool FUSED>
cudaError_t by_types(const StepLaunch &L, StepParamsPi &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32)
        return run<128, 16, KDA, kMaxTokens, __nv_bfloat16, float, FUSED>(P, s);
    if (L.in_dt == RS_BF16 && L.out_dt == RS_BF16)
        return run<128, 16, KDA, kMaxTokens, __nv_bfloat16, __nv_bfloat16, FUSED>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<128, 16, KDA, kMaxTokens, float, float, FUSED>(P, s);
    if (L.in_dt == RS_F16 && L.out_dt == RS_F32)
        return run<128, 16, KDA, kMaxTokens, __half, float, FUSED>(P, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_step_mixed_replay(const StepLaunch &L, StepParamsPi &P, cudaStream_t s) {
    if (L.D == 128 && L.khi == 16) {
        if (L.fused) return L.kda ? by_types<true, true>(L, P, s) : by_types<false, true>(L, P, s);
        return L.kda ? by_types<true, false>(L, P, s) : by_types<false, false>(L, P, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace rs
