// rs_ckpt_int8.cu -- dasc INT8 state checkpoint (sm_103a).
//
// dasc Appendix E.1 Eq. 8: the retained units of an FP32 state are quantised
// once when the checkpoint is written and dequantised once when it is reused:
// one FP32 scale per (layer, head, key channel) shared over dv -- one scale
// per state row here (rows = key channels) -- s = max(a, 1e-8)/127 from the
// row's absmax a, codes clip(rne(x/s), -127, 127), S^ = code * s.  The packed
// order is dasc's ragged Scheme 2 (§4.1, Appendix B): units of layer l at
// [o_{l-1}, o_l), a unit being a head (dk rows) or one key-channel row.
// Checkpoint slot: codes [o_L][rows][dv] int8, then scales [o_L][rows] f32,
// padded to 16 bytes.  Restore writes every row of the destination slot:
// retained rows dequantised, omitted rows +0.0 (dasc §4.2).
//
// One warp per state row (dv = 128: 16 bytes per lane); each warp keeps
// kRows rows in flight.  The absmax is a lane max plus one warp max-reduction
// (redux.sync), the scale is division-free (rs_quant.cuh), and the code is
// the exact RN(x/s) of the step kernels with the literal IEEE path for rows
// whose absmax is not finite -- the same values as the oracle's quantiser.
#include "rs_ckpt_int8.h"
#include "rs_quant.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

constexpr int kRows = 4;  // rows in flight per warp

template <int VPL> struct LaneVec;
template <> struct LaneVec<4> {
    float v[4];
    __device__ __forceinline__ void load(const uint8_t *p) {
        uint4 r;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                     : "l"(p));
        v[0] = __uint_as_float(r.x), v[1] = __uint_as_float(r.y), v[2] = __uint_as_float(r.z),
        v[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ void store(uint8_t *p) const {
        asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p),
                     "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                     "r"(__float_as_uint(v[3]))
                     : "memory");
    }
};
template <> struct LaneVec<2> {
    float v[2];
    __device__ __forceinline__ void load(const uint8_t *p) {
        uint2 r;
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
        v[0] = __uint_as_float(r.x), v[1] = __uint_as_float(r.y);
    }
    __device__ __forceinline__ void store(uint8_t *p) const {
        asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(__float_as_uint(v[0])),
                     "r"(__float_as_uint(v[1]))
                     : "memory");
    }
};

__device__ __forceinline__ float max_abs_nan2(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)));
    return r;
}

// code byte (two's complement) of x with scale s = -ns, reciprocal y = rcp_rn(s):
// RN(x/s) by two exact-remainder corrections, then round half to even.
__device__ __forceinline__ uint32_t code_of(float x, float ns, float y) {
    float t = __fmul_rn(x, y);
    t = __fmaf_rn(__fmaf_rn(t, ns, x), y, t);
    t = __fmaf_rn(__fmaf_rn(t, ns, x), y, t);
    return __float_as_uint(__fadd_rn(t, kRound)) & 0xffu;
}

template <int DV>
__global__ void __launch_bounds__(256) ckpt_pack_int8_kernel(const __grid_constant__ Int8CkptParams P,
                                                             uint32_t rows_per_pair) {
    constexpr int VPL = DV / 32;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.y;
    const int32_t ps = P.pool_slots[i], cs = P.ckpt_slots[i];
    const bool ps_ok = ps >= 0 && (int64_t)ps < P.n_pool_slots;
    const bool cs_ok = cs >= 0 && (int64_t)cs < P.n_ckpt_slots;
    if (!ps_ok || !cs_ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && P.status)
            atomicOr(P.status, (ps_ok ? 0 : RS_DEV_BAD_SLOT) | (cs_ok ? 0 : RS_DEV_BAD_CKPT_SLOT));
        return;
    }
    const uint32_t rmask = (1u << P.rows_log2) - 1u;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    uint8_t *ck = P.dst + (int64_t)cs * P.ckpt_slot_bytes;
    for (uint32_t base = warp * kRows; base < rows_per_pair; base += nwarps * kRows) {
        LaneVec<VPL> x[kRows];
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const uint32_t rr = base + k;
            if (rr < rows_per_pair) {
                const int32_t ku = __ldg(P.kept_unit + (rr >> P.rows_log2));
                const int64_t l = ku >> 20, u = ku & 0xfffff;
                x[k].load(P.src + l * P.layer_stride + (int64_t)ps * P.slot_bytes + u * P.unit_bytes +
                          (int64_t)(rr & rmask) * DV * 4 + lane * VPL * 4);
            }
        }
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const uint32_t rr = base + k;
            if (rr >= rows_per_pair) break;  // uniform over the warp
            float m = max_abs_nan2(x[k].v[0], x[k].v[1]);
            if constexpr (VPL == 4) m = max_abs_nan2(m, max_abs_nan2(x[k].v[2], x[k].v[3]));
            const float a = warp_max_abs_nan(m);
            const float sv = row_scale_from_absmax(a);
            uint32_t word = 0;
            if (a <= 3.402823466e38f) {  // finite absmax (uniform over the warp)
                const float y = __frcp_rn(sv), ns = -sv;
#pragma unroll
                for (int t = 0; t < VPL; ++t) word |= code_of(x[k].v[t], ns, y) << (8 * t);
            } else {  // inf or NaN in the row: the literal IEEE division
#pragma unroll
                for (int t = 0; t < VPL; ++t) word |= quant_exact(x[k].v[t], sv) << (8 * t);
            }
            uint8_t *crow = ck + (int64_t)rr * DV + lane * VPL;
            if constexpr (VPL == 4) *reinterpret_cast<uint32_t *>(crow) = word;
            else *reinterpret_cast<uint16_t *>(crow) = (uint16_t)word;
            if (lane == 0) *reinterpret_cast<float *>(ck + P.codes_bytes + (int64_t)rr * 4) = sv;
        }
    }
}

template <int DV>
__global__ void __launch_bounds__(256) ckpt_restore_int8_kernel(const __grid_constant__ Int8CkptParams P,
                                                                uint32_t rows_per_pair) {
    constexpr int VPL = DV / 32;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.y;
    const int32_t ps = P.pool_slots[i], cs = P.ckpt_slots[i];
    const bool ps_ok = ps >= 0 && (int64_t)ps < P.n_pool_slots;
    const bool cs_ok = cs >= 0 && (int64_t)cs < P.n_ckpt_slots;
    if (!ps_ok || !cs_ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && P.status)
            atomicOr(P.status, (ps_ok ? 0 : RS_DEV_BAD_SLOT) | (cs_ok ? 0 : RS_DEV_BAD_CKPT_SLOT));
        return;
    }
    const uint32_t rmask = (1u << P.rows_log2) - 1u;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const uint8_t *ck = P.src + (int64_t)cs * P.ckpt_slot_bytes;
    for (uint32_t base = warp * kRows; base < rows_per_pair; base += nwarps * kRows) {
        uint32_t word[kRows];
        float sc[kRows];
        uint8_t *dst[kRows];
        bool kept[kRows];
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const uint32_t rr = base + k;
            word[k] = 0;
            sc[k] = 0.0f;
            dst[k] = nullptr;
            kept[k] = false;
            if (rr < rows_per_pair) {
                const uint32_t u = rr >> P.rows_log2;
                const uint32_t l = u / (uint32_t)P.units_per_layer;
                const uint32_t x = u - l * (uint32_t)P.units_per_layer;
                const int32_t pidx = __ldg(P.all_pidx + u);
                dst[k] = P.dst + (int64_t)l * P.layer_stride + (int64_t)ps * P.slot_bytes +
                         (int64_t)x * P.unit_bytes + (int64_t)(rr & rmask) * DV * 4 + lane * VPL * 4;
                if (pidx >= 0) {
                    const int64_t crow = ((int64_t)pidx << P.rows_log2) + (rr & rmask);
                    kept[k] = true;
                    if constexpr (VPL == 4) word[k] = __ldg(reinterpret_cast<const uint32_t *>(ck + crow * DV) + lane);
                    else word[k] = __ldg(reinterpret_cast<const uint16_t *>(ck + crow * DV) + lane);
                    sc[k] = __ldg(reinterpret_cast<const float *>(ck + P.codes_bytes) + crow);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            if (!dst[k]) break;
            LaneVec<VPL> y;
            const uint32_t w = word[k] ^ 0x80808080u;
#pragma unroll
            for (int t = 0; t < VPL; ++t) {
                const float c = __fadd_rn(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540 + t)), -kCodeBias);
                y.v[t] = kept[k] ? __fmul_rn(c, sc[k]) : 0.0f;
            }
            y.store(dst[k]);
        }
    }
}

template <bool PACK> cudaError_t launch(const Int8CkptParams &P, cudaStream_t s) {
    if (P.dv != 64 && P.dv != 128) return cudaErrorNotSupported;
    const int64_t rows = (PACK ? P.n_kept : P.n_all) << P.rows_log2;
    if (rows >= (1ll << 31) || P.n > 65535) return cudaErrorNotSupported;
    if (rows == 0 || P.n == 0) return cudaSuccess;
    const int64_t warps_needed = (rows + kRows - 1) / kRows;
    int64_t bx = (warps_needed * 32 + 255) / 256;
    // CTAs of 8 warps per SM over the whole grid: 8 for pack, 16 for restore
    // (restore's writes are the larger side; measured faster with more warps)
    const int64_t per_sm = PACK ? 8 : 16;
    int64_t cap = ((int64_t)device_sm_count() * per_sm + P.n - 1) / P.n;
    if (cap < 1) cap = 1;
    if (bx > cap) bx = cap;
    dim3 grid((unsigned)bx, (unsigned)P.n);
    if (PACK) {
        if (P.dv == 128) ckpt_pack_int8_kernel<128><<<grid, 256, 0, s>>>(P, (uint32_t)rows);
        else ckpt_pack_int8_kernel<64><<<grid, 256, 0, s>>>(P, (uint32_t)rows);
    } else {
        if (P.dv == 128) ckpt_restore_int8_kernel<128><<<grid, 256, 0, s>>>(P, (uint32_t)rows);
        else ckpt_restore_int8_kernel<64><<<grid, 256, 0, s>>>(P, (uint32_t)rows);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ckpt_pack_int8(const Int8CkptParams &P, cudaStream_t s) { return launch<true>(P, s); }
cudaError_t launch_ckpt_restore_int8(const Int8CkptParams &P, cudaStream_t s) { return launch<false>(P, s); }

}  // namespace rs
