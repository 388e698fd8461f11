// rs_damp_convert.cu -- FP32 <-> DAMP-exact mixed state conversion (DAMP
// Appendix A.1, A.3 Eq. 17, A.4).  FP32 -> DAMP: physical row r takes logical
// key channel pi[r], each value is divided by its value-scaling factor c'_v,
// FP16 rows round to nearest even and INT8 rows are quantised in groups of 32
// values (one warp per group: the absmax is one warp max-reduction) with the
// literal IEEE quotient, or with the fused arithmetic's one-rounding product
// x * RN(1/s) when the destination layout asks for it (groups whose absmax is
// inf or NaN keep the quotient).  DAMP -> FP32: dequantise, multiply by c'_v, write the
// logical row.  One CTA of D threads per (slot, head), thread v on column v.
// Used to initialise and inspect pools, not on the decode path.
#include "rs_damp.h"
#include "rs_step.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

template <int D, int KH, bool FUSED>
__global__ void __launch_bounds__(D) damp_convert_kernel(const __grid_constant__ ConvertParamsDamp P) {
    constexpr int NG = D / kDampGroup;
    constexpr int kBytes = 2 * KH * D + (D - KH) * D + 4 * (D - KH) * NG;
    __shared__ __align__(16) uint8_t tile_s[kBytes];
    __shared__ uint8_t pi_s[D];
    const int tid = threadIdx.x, lane = tid & 31, grp = tid / kDampGroup;
    const int i = blockIdx.x / P.Hv, h = blockIdx.x - (blockIdx.x / P.Hv) * P.Hv;
    const int32_t slot = P.slots[i];
    if (slot < 0 || (int64_t)slot >= P.n_slots) {
        if (tid == 0 && P.status) atomicOr(P.status, RS_DEV_BAD_SLOT);
        return;
    }
    pi_s[tid] = P.pi[h * D + tid];
    const float c = P.cs[h * D + tid];
    __syncthreads();
    const size_t tile = (size_t)slot * P.Hv + h;
    uint16_t *hi = reinterpret_cast<uint16_t *>(tile_s);
    uint8_t *lo = tile_s + 2 * KH * D;
    float *sc = reinterpret_cast<float *>(tile_s + 2 * KH * D + (D - KH) * D);
    if (P.to_mixed) {
        const float *src = static_cast<const float *>(P.src) + tile * (D * D);
        for (int r = 0; r < D; ++r) {
            const float x = __fdiv_rn(src[(int)pi_s[r] * D + tid], c);
            if (r < KH) {
                const __half hv = __float2half_rn(x);
                hi[((r / 2) * D + tid) * 2 + (r % 2)] = *reinterpret_cast<const uint16_t *>(&hv);
            } else {
                const int q = r - KH;
                const float a = warp_max_abs_nan(x);  // one group = one warp
                const float s = __fdiv_rn(fmaxf(a, 1e-8f), 127.0f);
                uint32_t code;
                if constexpr (FUSED) code = quant_rcp_or_exact(x, s, a <= 3.402823466e38f ? __frcp_rn(s) : 0.0f);
                else code = quant_exact(x, s);
                lo[((q / 4) * D + tid) * 4 + (q % 4)] = (uint8_t)code;
                if (lane == 0) sc[q * NG + grp] = s;
            }
        }
        __syncthreads();
        uint4 *dst4 = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.dst) + tile * kBytes);
        const uint4 *src4 = reinterpret_cast<const uint4 *>(tile_s);
        for (int j = tid; j < kBytes / 16; j += D) dst4[j] = src4[j];
    } else {
        const uint8_t *src = static_cast<const uint8_t *>(P.src) + tile * kBytes;
        const uint16_t *hig = reinterpret_cast<const uint16_t *>(src);
        const int8_t *log = reinterpret_cast<const int8_t *>(src + 2 * KH * D);
        const float *scg = reinterpret_cast<const float *>(src + 2 * KH * D + (D - KH) * D);
        float *dst = static_cast<float *>(P.dst) + tile * (D * D);
        for (int r = 0; r < D; ++r) {
            float x;
            if (r < KH) {
                const uint16_t b = hig[((r / 2) * D + tid) * 2 + (r % 2)];
                x = __half2float(*reinterpret_cast<const __half *>(&b));
            } else {
                const int q = r - KH;
                x = __fmul_rn((float)log[((q / 4) * D + tid) * 4 + (q % 4)], scg[q * NG + grp]);
            }
            dst[(int)pi_s[r] * D + tid] = __fmul_rn(x, c);
        }
    }
}

}  // namespace

cudaError_t launch_convert_damp(int D, int khi, ConvertParamsDamp &P, cudaStream_t s) {
    if (P.n == 0) return cudaSuccess;
    const unsigned grid = (unsigned)P.n * (unsigned)P.Hv;
    if (D == 128 && khi == 16) {
        if (P.fused) damp_convert_kernel<128, 16, true><<<grid, 128, 0, s>>>(P);
        else damp_convert_kernel<128, 16, false><<<grid, 128, 0, s>>>(P);
    } else {
        return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace rs
