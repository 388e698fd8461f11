// rs_step_mixed_decode.cu -- single decode steps on the mixed FP16/INT8
// layout (dk = dv = 128, 16 FP16 rows per head): a warp pair per tile over a
// ring of shared-memory stages (rs_mixed_decode.cuh).
#include "rs_mixed_decode.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

// warps per tile: 2 (two columns per lane, 16 warps per CTA) or 1 (four)
constexpr int kMixedWpt = 2;
constexpr int kMixedSlots = 8;  // tile slots per CTA

template <int D, int KHI, bool KDA, typename TI, typename TO, bool FUSED>
cudaError_t run(StepParamsPi &P, cudaStream_t s) {
    using Sh = MixedWarpShape<D, KHI, KDA, TI, kMixedWpt, FUSED>;
    auto kern = mixed_decode_kernel<D, KHI, KDA, TI, TO, kMixedWpt, FUSED>;
    const int header = Sh::kHeader + (P.Hv * D + 127) / 128 * 128;
    const int smax = device_max_smem_optin();
    // NSLOT tile slots and a ring of NS > NSLOT stages in the shared memory there is
    int NSLOT = kMixedSlots, NS = 0;
    for (; NSLOT >= 1; --NSLOT) {
        const int avail = smax - header - NSLOT * Sh::kSlotBytes;
        NS = avail > 0 ? avail / Sh::kStage : 0;
        if (NS > kMixedMaxStages) NS = kMixedMaxStages;
        if (NS >= NSLOT + 1) break;
    }
    if (NSLOT < 1) return cudaErrorNotSupported;
    const int W = NSLOT * kMixedWpt;
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
    return launch_pdl(kern, dim3(grid), dim3(W * 32), smem, s, P);
}

template <bool KDA, bool FUSED>
cudaError_t by_types(const StepLaunch &L, StepParamsPi &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32) return run<128, 16, KDA, __nv_bfloat16, float, FUSED>(P, s);
    if (L.in_dt == RS_BF16 && L.out_dt == RS_BF16)
        return run<128, 16, KDA, __nv_bfloat16, __nv_bfloat16, FUSED>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<128, 16, KDA, float, float, FUSED>(P, s);
    if (L.in_dt == RS_F16 && L.out_dt == RS_F32) return run<128, 16, KDA, __half, float, FUSED>(P, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_step_mixed_decode(const StepLaunch &L, StepParamsPi &P, cudaStream_t s) {
    if (L.D == 128 && L.khi == 16) {
        if (L.fused) return L.kda ? by_types<true, true>(L, P, s) : by_types<false, true>(L, P, s);
        return L.kda ? by_types<true, false>(L, P, s) : by_types<false, false>(L, P, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace rs
