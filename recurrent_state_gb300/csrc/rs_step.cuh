// rs_step.cuh -- decode-step and speculative-replay kernel (sm_103a).
//
// One "group" of D threads (D = dk = dv) advances one state tile (sequence b,
// value head h) at a time; a CTA holds G groups and the grid is persistent,
// each group walking the tiles b*Hv+h in a fixed stride.  Thread v of a group
// owns column v of the tile: its D values live in registers for the whole
// step (or the whole replay), so
//   * the two reductions over key channels (p = S^T k, o = S^T q) are
//     sequential FMA chains in ascending row order inside one thread, which
//     reproduces the oracle's FP32 evaluation order exactly;
//   * the decay and the rank-1 write are elementwise on registers;
//   * a replay keeps the state on chip across tokens ("Serving recurrent
//     attention", speculative decoding without state snapshots).
// The tile and the token inputs arrive through a 1-D bulk TMA copy
// (cp.async.bulk + mbarrier) into the group's shared-memory stage; as soon as
// the stage has been read into registers the group issues the copy of its
// next tile, so HBM reads of tile i+1 overlap the arithmetic of tile i.
// Results go straight from registers to HBM with coalesced stores (a warp
// writes 32 consecutive columns of a row).
//
// Mixed layout (DAMP §5.2, Appendix A.4): FP16 rows and INT8 rows with one
// FP32 scale per row are dequantised into the registers, updated in FP32, and
// requantised in the same pass; the per-row absmax is a warp max-reduction
// (redux.sync) plus a 4-warp combine in shared memory.  The INT8 code is
// round_half_even(x / s) with x / s the IEEE quotient: the kernel computes
// q0 = x * rcp_rn(s); since |q0 - fl(x/s)| <= 3 * 2^-24 * |x/s| < 2^-15 for
// |x/s| <= 127.0001, every q0 farther than 2^-15 from a half-integer rounds
// like fl(x/s); the rest (about 6e-5 of the values) take the exact IEEE
// division.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rs_device.cuh"
#include "rs_internal.h"

namespace rs {

template <int D, int KHI, bool KDA, typename TI>
struct StepShape {
    static constexpr bool kMixed = KHI >= 0;
    static constexpr int kKhi = KHI < 0 ? 0 : KHI;
    static constexpr int kStateBytes =
        kMixed ? (2 * kKhi * D + (D - kKhi) * D + 4 * (D - kKhi)) : D * D * 4;
    static constexpr int kStatePad = (kStateBytes + 127) / 128 * 128;
    static constexpr int kVecBytes = D * (int)sizeof(TI);
    static constexpr int kTokBytes = 3 * kVecBytes + (KDA ? D * 4 : 0);  // k, q, v, alpha
    static constexpr int kWarps = D / 32;
    // per-token row vectors in shared memory: K, BK, Q, V (+ A for KDA), floats
    static constexpr int kRowVecs = KDA ? 5 : 4;

    static constexpr int region_bytes(int T) {
        int r = kStatePad + T * kTokBytes;
        r = (r + 127) / 128 * 128;
        r += T * kRowVecs * D * 4;
        if (kMixed) r += kWarps * D * 4 + D * 8;  // absmax partials, (scale, recip)
        return (r + 127) / 128 * 128;
    }
};

__device__ __forceinline__ void report(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// INT8 code of x for a row with scale s and y = rcp_rn(s) (y == 0 marks a
// row whose absmax is not finite: every value there takes the exact path).
__device__ __forceinline__ uint32_t quant_code(float x, float s, float y) {
    if (y != 0.0f) {
        const float q0 = __fmul_rn(x, y);
        const float m = __fadd_rn(q0, 12582912.0f);  // 1.5 * 2^23: rounds q0 half-to-even
        const float t = __fsub_rn(q0, __fsub_rn(m, 12582912.0f));
        if (fabsf(t) < 0.499969482421875f)  // 0.5 - 2^-15
            return __float_as_uint(m);      // low byte = two's complement code
    }
    float r = rintf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<uint32_t>(static_cast<int32_t>(r));
}


// Requantise the FP32 column x (thread tid of a group of D threads, warp wig,
// lane lane) into a mixed-layout tile in global memory: FP16 rows
// 0..KH-1, INT8 rows KH..D-1 with one FP32 scale per row.  red ([D/32][D]
// floats) and sy ([D] float2) are group-private shared scratch; bar_id/D name
// the group barrier.  Matches the oracle's quantiser bit for bit.
template <int D, int KH>
__device__ __forceinline__ void mixed_requant_store(const float (&x)[D], uint8_t *tile, float *red,
                                                    float2 *sy, int tid, int lane, int wig,
                                                    uint32_t bar_id) {
    constexpr int W = D / 32;
    // per-row absmax: warp reduction, then combine the group's warps
#pragma unroll
    for (int r = KH; r < D; ++r) {
        const float m = warp_max_abs_nan(x[r]);
        if (lane == 0) red[wig * D + r] = m;
    }
    group_sync(bar_id, D);
    if (tid >= KH) {
        uint32_t ab = __float_as_uint(red[tid]);
#pragma unroll
        for (int w = 1; w < W; ++w) ab = max(ab, __float_as_uint(red[w * D + tid]));
        const float a = __uint_as_float(ab);  // >= 0, or NaN (largest bit pattern)
        const float s = __fdiv_rn(fmaxf(a, 1e-8f), 127.0f);
        const bool finite = ab < 0x7f800000u;
        sy[tid] = make_float2(s, finite ? __frcp_rn(s) : 0.0f);
        reinterpret_cast<float *>(tile + 2 * KH * D + (D - KH) * D)[tid - KH] = s;
    }
    group_sync(bar_id, D);
    __half *hi = reinterpret_cast<__half *>(tile);
#pragma unroll
    for (int r = 0; r < KH; ++r) hi[r * D + tid] = __float2half_rn(x[r]);
    uint8_t *lo = tile + 2 * KH * D;
#pragma unroll
    for (int r = KH; r < D; ++r) {
        const float2 v2 = sy[r];
        lo[(r - KH) * D + tid] = static_cast<uint8_t>(quant_code(x[r], v2.x, v2.y) & 0xffu);
    }
}

// Dequantise column tid of a mixed-layout tile (shared or global memory).
template <int D, int KH>
__device__ __forceinline__ void mixed_dequant(const uint8_t *tile, int tid, float (&x)[D]) {
    const __half *hi = reinterpret_cast<const __half *>(tile);
    const int8_t *lo = reinterpret_cast<const int8_t *>(tile + 2 * KH * D);
    const float *sc = reinterpret_cast<const float *>(tile + 2 * KH * D + (D - KH) * D);
#pragma unroll
    for (int r = 0; r < KH; ++r) x[r] = __half2float(hi[r * D + tid]);
#pragma unroll
    for (int r = KH; r < D; ++r) x[r] = __fmul_rn(static_cast<float>(lo[(r - KH) * D + tid]), sc[r - KH]);
}

template <int D, int KHI, bool KDA, int MAXT, typename TI, typename TO, typename PT>
__global__ void __launch_bounds__(kStepThreads, 1)
    step_kernel(const __grid_constant__ PT P) {
    using S = StepShape<D, KHI, KDA, TI>;
    constexpr bool MIXED = S::kMixed;
    constexpr int KH = S::kKhi;

    extern __shared__ __align__(128) uint8_t smem[];
    const int G = blockDim.x / D;
    const int grp = threadIdx.x / D;
    const int tid = threadIdx.x - grp * D;  // column v; also row u when staging rows
    const int lane = threadIdx.x & 31;
    const int wig = tid >> 5;               // warp within the group
    const int T = P.T_max;
    const int Hv = P.Hv, Hk = P.Hk;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *pi_s = smem + 128;
    uint8_t *region = smem + P.header_bytes + (size_t)grp * P.region_bytes;
    uint8_t *stage = region;
    float *rowv = reinterpret_cast<float *>(region + ((S::kStatePad + T * S::kTokBytes + 127) / 128 * 128));
    // rowv layout per token t: [K | BK | Q | V | A?] each D floats
    float *red = rowv + T * S::kRowVecs * D;          // [kWarps][D]      (mixed)
    float2 *sy = reinterpret_cast<float2 *>(red + S::kWarps * D);  // [D] (mixed)

    if (threadIdx.x < G) mbar_init(&bars[threadIdx.x], 1);
    if constexpr (MIXED)
        for (int i = threadIdx.x; i < Hv * D; i += blockDim.x) pi_s[i] = P.pi[i];
    fence_mbar_init();
    __syncthreads();

    uint64_t *bar = &bars[grp];
    const uint32_t bar_id = 1 + grp;
    const int items = P.B * Hv;
    const int gstride = gridDim.x * G;
    const TI *q_g = static_cast<const TI *>(P.q);
    const TI *k_g = static_cast<const TI *>(P.k);
    const TI *v_g = static_cast<const TI *>(P.v);
    uint8_t *pool = static_cast<uint8_t *>(P.pool);

    // Producer step, run by thread 0 of the group: start the copies of item it.
    auto issue = [&](int it) {
        if (it >= items) return;
        const int b = it / Hv, h = it - (it / Hv) * Hv;
        const int32_t slot = P.slot_idx[b];
        const int32_t n = P.replay ? P.n_accept[b] : 1;
        if (slot < 0 || (int64_t)slot >= P.n_slots || n <= 0 || n > T) return;
        const int g = h / (Hv / Hk);
        mbar_arrive_expect_tx(bar, (uint32_t)(S::kStateBytes + n * S::kTokBytes));
        bulk_g2s(stage, pool + ((size_t)slot * Hv + h) * S::kStateBytes, S::kStateBytes, bar);
        for (int t = 0; t < n; ++t) {
            uint8_t *tb = stage + S::kStatePad + t * S::kTokBytes;
            const size_t bt = (size_t)b * T + t;
            bulk_g2s(tb, k_g + (bt * Hk + g) * D, S::kVecBytes, bar);
            bulk_g2s(tb + S::kVecBytes, q_g + (bt * Hk + g) * D, S::kVecBytes, bar);
            bulk_g2s(tb + 2 * S::kVecBytes, v_g + (bt * Hv + h) * D, S::kVecBytes, bar);
            if (KDA) bulk_g2s(tb + 3 * S::kVecBytes, P.alpha + (bt * Hv + h) * D, D * 4, bar);
        }
    };

    int item = blockIdx.x * G + grp;
    if (tid == 0) issue(item);
    uint32_t phase = 0;

    for (; item < items; item += gstride) {
        const int b = item / Hv, h = item - (item / Hv) * Hv;
        const int32_t slot = P.slot_idx[b];
        const int32_t n = P.replay ? P.n_accept[b] : 1;
        const bool slot_ok = slot >= 0 && (int64_t)slot < P.n_slots;
        const bool n_ok = n >= 0 && n <= T;
        if (!slot_ok || !n_ok || n == 0) {
            if (tid == 0) {
                if (!slot_ok) report(P.status, 1);
                else if (!n_ok) report(P.status, 2);
                issue(item + gstride);
            }
            continue;
        }
        // Scalars of this item, loaded before the wait so their latency hides.
        float beta_r[MAXT], alpha_r[MAXT];
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
            beta_r[t] = 0.0f;
            alpha_r[t] = 0.0f;
            if (t < n) {
                const size_t bt = (size_t)b * T + t;
                beta_r[t] = P.beta[bt * Hv + h];
                if (!KDA) alpha_r[t] = P.alpha[bt * Hv + h];
            }
        }

        bool got = mbar_wait_bounded(bar, phase);
        if (!got) got = mbar_wait_bounded(bar, phase);  // copies still in flight get a second bound
        if (group_sync_or(bar_id, D, !got)) {
            if (tid == 0) report(P.status, 8);
            return;
        }
        phase ^= 1u;

        // ---- state tile -> registers --------------------------------------
        float x[D];
        if constexpr (!MIXED) {
            const float *st = reinterpret_cast<const float *>(stage);
#pragma unroll
            for (int u = 0; u < D; ++u) x[u] = st[u * D + tid];
        } else {
            mixed_dequant<D, KH>(stage, tid, x);
        }

        // ---- token inputs -> per-row vectors (row u built by thread u) -----
        const int src = MIXED ? (int)pi_s[h * D + tid] : tid;
        for (int t = 0; t < n; ++t) {
            const uint8_t *tb = stage + S::kStatePad + t * S::kTokBytes;
            const TI *kt = reinterpret_cast<const TI *>(tb);
            const TI *qt = reinterpret_cast<const TI *>(tb + S::kVecBytes);
            const TI *vt = reinterpret_cast<const TI *>(tb + 2 * S::kVecBytes);
            float *rv = rowv + t * S::kRowVecs * D;
            const float kf = load_as_f32<TI>(kt + src);
            float bt = 0.0f;
#pragma unroll
            for (int tt = 0; tt < MAXT; ++tt)
                if (tt == t) bt = beta_r[tt];
            rv[tid] = kf;
            rv[D + tid] = __fmul_rn(bt, kf);
            rv[2 * D + tid] = load_as_f32<TI>(qt + src);
            rv[3 * D + tid] = load_as_f32<TI>(vt + tid);  // value coordinates: no row map
            if (KDA) rv[4 * D + tid] = reinterpret_cast<const float *>(tb + 3 * S::kVecBytes)[src];
        }
        group_sync(bar_id, D);  // stage fully read, row vectors visible

        if (tid == 0) {
            fence_proxy_async_smem();
            issue(item + gstride);  // the stage now belongs to the next tile
        }

        // ---- the recurrence, token by token, state in registers -----------
        for (int t = 0; t < n; ++t) {
            const float *rv = rowv + t * S::kRowVecs * D;
            float a_s = 0.0f;
#pragma unroll
            for (int tt = 0; tt < MAXT; ++tt)
                if (tt == t) a_s = alpha_r[tt];
            // S <- diag(alpha) S ;  p = S^T k  (ascending rows)
            float p = 0.0f;
#pragma unroll
            for (int u = 0; u < D; u += 4) {
                const float4 kk = *reinterpret_cast<const float4 *>(rv + u);
                float4 aa;
                if (KDA) aa = *reinterpret_cast<const float4 *>(rv + 4 * D + u);
                else aa = make_float4(a_s, a_s, a_s, a_s);
                x[u + 0] = __fmul_rn(x[u + 0], aa.x);
                p = __fmaf_rn(x[u + 0], kk.x, p);
                x[u + 1] = __fmul_rn(x[u + 1], aa.y);
                p = __fmaf_rn(x[u + 1], kk.y, p);
                x[u + 2] = __fmul_rn(x[u + 2], aa.z);
                p = __fmaf_rn(x[u + 2], kk.z, p);
                x[u + 3] = __fmul_rn(x[u + 3], aa.w);
                p = __fmaf_rn(x[u + 3], kk.w, p);
            }
            const float e = __fsub_rn(rv[3 * D + tid], p);
            // S <- S + beta k e^T ;  o = S^T q  (ascending rows)
            float o = 0.0f;
#pragma unroll
            for (int u = 0; u < D; u += 4) {
                const float4 bk = *reinterpret_cast<const float4 *>(rv + D + u);
                const float4 qq = *reinterpret_cast<const float4 *>(rv + 2 * D + u);
                x[u + 0] = __fmaf_rn(bk.x, e, x[u + 0]);
                o = __fmaf_rn(x[u + 0], qq.x, o);
                x[u + 1] = __fmaf_rn(bk.y, e, x[u + 1]);
                o = __fmaf_rn(x[u + 1], qq.y, o);
                x[u + 2] = __fmaf_rn(bk.z, e, x[u + 2]);
                o = __fmaf_rn(x[u + 2], qq.z, o);
                x[u + 3] = __fmaf_rn(bk.w, e, x[u + 3]);
                o = __fmaf_rn(x[u + 3], qq.w, o);
            }
            if (P.o) {
                TO *og = static_cast<TO *>(P.o);
                store_from_f32<TO>(og + (((size_t)b * T + t) * Hv + h) * D + tid, o);
            }
        }

        // ---- registers -> HBM ---------------------------------------------
        uint8_t *tile = pool + ((size_t)slot * Hv + h) * S::kStateBytes;
        if constexpr (!MIXED) {
            float *st = reinterpret_cast<float *>(tile);
#pragma unroll
            for (int u = 0; u < D; ++u) st[u * D + tid] = x[u];
        } else {
            mixed_requant_store<D, KH>(x, tile, red, sy, tid, lane, wig, bar_id);
        }
        group_sync(bar_id, D);  // row vectors / partials free for the next item
    }
}

}  // namespace rs
