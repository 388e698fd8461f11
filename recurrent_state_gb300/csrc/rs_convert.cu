// rs_convert.cu -- FP32 <-> mixed FP16/INT8 state conversion (DAMP §5.2,
// Appendix A.3 Eq. 17, Appendix A.4), and same-layout slot copies.
//
// One CTA of D threads per (slot, head) tile; thread v owns column v.
// FP32 -> mixed: physical row r of the mixed tile takes logical key channel
// pi[r]; the rows are requantised by the same routine as the replay kernel,
// in the IEEE or the fused arithmetic of the destination layout.
// Mixed -> FP32: dequantise and write each physical row back to its logical
// channel.  Used to initialise and inspect mixed pools, not on the decode path.
#include "rs_step.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

template <int D, int KH, bool FUSED>
__global__ void __launch_bounds__(D) convert_kernel(const __grid_constant__ ConvertParamsPi P) {
    constexpr int kMixedBytes = 2 * KH * D + (D - KH) * D + 4 * (D - KH);
    __shared__ float red[(D / 32) * D];
    __shared__ __align__(16) float scl[D];
    __shared__ __align__(16) float nscl[D];
    __shared__ __align__(16) float rcp[D];
    __shared__ int flag;
    __shared__ __align__(16) uint8_t out[kMixedBytes];
    __shared__ uint8_t pi_s[D];
    const int tid = threadIdx.x, lane = tid & 31, wig = tid >> 5;
    const int i = blockIdx.x / P.Hv, h = blockIdx.x - (blockIdx.x / P.Hv) * P.Hv;
    const int32_t slot = P.slots[i];
    if (slot < 0 || (int64_t)slot >= P.n_slots) {
        if (tid == 0 && P.status) atomicOr(P.status, RS_DEV_BAD_SLOT);
        return;
    }
    pi_s[tid] = P.pi[h * D + tid];
    if (tid == 0) flag = 0;
    __syncthreads();
    const size_t tile = (size_t)slot * P.Hv + h;
    float2 x[D / 2];
    if (P.to_mixed) {
        const float *src = static_cast<const float *>(P.src) + tile * (D * D);
#pragma unroll
        for (int j = 0; j < D / 2; ++j)
            x[j] = make_float2(src[(int)pi_s[2 * j] * D + tid], src[(int)pi_s[2 * j + 1] * D + tid]);
        mixed_requant_smem<D, KH, FUSED>(x, out, red, scl, nscl, rcp, &flag, tid, lane, wig, 0, [] {});
        __syncthreads();
        uint4 *dst4 = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.dst) + tile * kMixedBytes);
        const uint4 *src4 = reinterpret_cast<const uint4 *>(out);
        for (int j = tid; j < kMixedBytes / 16; j += D) dst4[j] = src4[j];
    } else {
        mixed_dequant<D, KH>(static_cast<const uint8_t *>(P.src) + tile * kMixedBytes, tid, x);
        float *dst = static_cast<float *>(P.dst) + tile * (D * D);
#pragma unroll
        for (int j = 0; j < D / 2; ++j) {
            dst[(int)pi_s[2 * j] * D + tid] = x[j].x;
            dst[(int)pi_s[2 * j + 1] * D + tid] = x[j].y;
        }
    }
}

// Same-layout copy of whole heads: 16-byte vectors, one CTA per (slot, head).
__global__ void copy_heads_kernel(const uint8_t *src, uint8_t *dst, int64_t head_bytes,
                                  const int32_t *slots, int64_t n_slots, int32_t Hv,
                                  int32_t *status) {
    const int i = blockIdx.x / Hv, h = blockIdx.x - (blockIdx.x / Hv) * Hv;
    const int32_t slot = slots[i];
    if (slot < 0 || (int64_t)slot >= n_slots) {
        if (threadIdx.x == 0 && status) atomicOr(status, RS_DEV_BAD_SLOT);
        return;
    }
    const size_t off = ((size_t)slot * Hv + h) * head_bytes;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + off);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst + off);
    for (int64_t j = threadIdx.x; j < head_bytes / 16; j += blockDim.x) d4[j] = s4[j];
}

}  // namespace

cudaError_t launch_convert(int D, int khi, ConvertParamsPi &P, cudaStream_t s) {
    if (P.n == 0) return cudaSuccess;
    const unsigned grid = (unsigned)P.n * (unsigned)P.Hv;
    if (D == 128 && khi == 16) {
        if (P.fused) convert_kernel<128, 16, true><<<grid, 128, 0, s>>>(P);
        else convert_kernel<128, 16, false><<<grid, 128, 0, s>>>(P);
        return cudaGetLastError();
    }
    return cudaErrorNotSupported;
}

cudaError_t launch_copy_heads(const void *src, void *dst, int64_t head_bytes, const int32_t *slots,
                              int32_t n, int64_t n_slots, int32_t Hv, int32_t *status,
                              cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    copy_heads_kernel<<<(unsigned)n * (unsigned)Hv, 256, 0, s>>>(
        static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), head_bytes, slots, n_slots,
        Hv, status);
    return cudaGetLastError();
}

}  // namespace rs
