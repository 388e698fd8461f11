// rs_step_damp_decode.cu -- single decode steps on the DAMP-exact mixed
// layout (dk = dv = 128, 16 FP16 rows, INT8 groups of 32, value scaling):
// a warp pair per tile over a ring of shared-memory stages (rs_damp_decode.cuh).
#include "rs_damp_decode.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

constexpr int kDampSlots = 8;  // tile slots (warp pairs) per CTA

template <int D, int KHI, bool KDA, typename TI, typename TO, bool FUSED>
cudaError_t run(StepParamsDamp &P, cudaStream_t s) {
    using Sh = DampShape<D, KHI, KDA, TI>;
    auto kern = damp_decode_kernel<D, KHI, KDA, TI, TO, FUSED>;
    const int header = Sh::kHeader + (P.Hv * D + 127) / 128 * 128;
    const int smax = device_max_smem_optin();
    int NSLOT = kDampSlots, NS = 0;
    for (; NSLOT >= 1; --NSLOT) {
        const int avail = smax - header - NSLOT * Sh::kSlotBytes;
        NS = avail > 0 ? avail / Sh::kStage : 0;
        if (NS > kMixedMaxStages) NS = kMixedMaxStages;
        if (NS >= NSLOT + 1) break;
    }
    if (NSLOT < 1) return cudaErrorNotSupported;
    const int items = P.B * P.Hv;
    int grid = device_sm_count();
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    P.header_bytes = header;
    P.region_bytes = Sh::kStage;
    P.stages = NS;
    const int smem = header + NSLOT * Sh::kSlotBytes + NS * Sh::kStage;
    cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(NSLOT * 64), smem, s, P);
}

template <bool KDA, bool FUSED>
cudaError_t by_types(const StepLaunch &L, StepParamsDamp &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32) return run<128, 16, KDA, __nv_bfloat16, float, FUSED>(P, s);
    if (L.in_dt == RS_BF16 && L.out_dt == RS_BF16)
        return run<128, 16, KDA, __nv_bfloat16, __nv_bfloat16, FUSED>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<128, 16, KDA, float, float, FUSED>(P, s);
    if (L.in_dt == RS_F16 && L.out_dt == RS_F32) return run<128, 16, KDA, __half, float, FUSED>(P, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_step_damp_decode(const StepLaunch &L, StepParamsDamp &P, cudaStream_t s) {
    if (L.D == 128 && L.khi == 16) {
        if (L.fused) return L.kda ? by_types<true, true>(L, P, s) : by_types<false, true>(L, P, s);
        return L.kda ? by_types<true, false>(L, P, s) : by_types<false, false>(L, P, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace rs
