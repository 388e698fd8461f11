// rs_step_f32_d128.cu -- instantiations of the step kernel for the FP32 layout, dk = dv = 128.
#include "rs_step.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

template <int D, bool KDA, int MAXT, typename TI, typename TO>
cudaError_t run(StepParams &P, cudaStream_t s) {
    using Sh = StepShape<D, -1, KDA, TI>;
    auto kern = step_kernel<D, -1, KDA, MAXT, TI, TO, StepParams>;
    const int region = Sh::region_bytes(P.T_max);
    const int header = 128;
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

template <int D, bool KDA, int MAXT>
cudaError_t by_types(const StepLaunch &L, StepParams &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32) return run<D, KDA, MAXT, __nv_bfloat16, float>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<D, KDA, MAXT, float, float>(P, s);
    if (L.in_dt == RS_F16 && L.out_dt == RS_F32) return run<D, KDA, MAXT, __half, float>(P, s);
    if (D == 128 && L.in_dt == RS_BF16 && L.out_dt == RS_BF16)
        return run<D, KDA, MAXT, __nv_bfloat16, __nv_bfloat16>(P, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_step_f32_d128(const StepLaunch &L, StepParams &P, cudaStream_t s) {
    const bool multi = P.T_max > 1 || P.replay;
    if (L.D == 128) {
        if (multi) return L.kda ? by_types<128, true, kMaxTokens>(L, P, s) : by_types<128, false, kMaxTokens>(L, P, s);
        return L.kda ? by_types<128, true, 1>(L, P, s) : by_types<128, false, 1>(L, P, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace rs
