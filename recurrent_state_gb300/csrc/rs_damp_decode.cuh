// rs_damp_decode.cuh -- single-token decode on the DAMP-exact mixed layout:
// FP16 rows, INT8 rows with one FP32 scale per group of 32 values along dv,
// and value scaling (DAMP Appendix A.1, A.3 Eq. 18, A.4 "Fused decoding").
//
// Same pipeline as rs_mixed_decode.cuh (two warps per tile, a ring of
// shared-memory stages, the new words stored from registers to HBM), with the columns
// of a lane chosen so that a scale group is one warp: lane l of tile warp t
// owns columns 64t + l and 64t + 32 + l, i.e. one column of group 2t and one
// of group 2t + 1.  A group's row maximum is then one warp max-reduction
// (redux.sync) and no partial maxima cross warps.  The value-scaling factors
// c'_v enter as v' = v / c' before the prediction error and o = c' o' after
// the readout chain.  Every value is computed with the same operations in the
// same order as the oracle's transformed step.
// Fused arithmetic (FUSED): each new code is one fused multiply-add, the
// integer nearest to x * RN(1/s); the step itself is the same.
#pragma once

#include "rs_damp.h"
#include "rs_mixed_decode.cuh"

namespace rs {

template <int D, int KH, bool KDA, typename TI>
struct DampShape {
    static constexpr int kGroups = D / kDampGroup;
    static constexpr int kStateBytes = 2 * KH * D + (D - KH) * D + 4 * (D - KH) * kGroups;
    static constexpr int kStatePad = (kStateBytes + 127) / 128 * 128;
    static constexpr int kVecBytes = D * (int)sizeof(TI);
    static constexpr int kTokBytes = 3 * kVecBytes + (KDA ? D * 4 : 0);
    static constexpr int kStage = (kStatePad + kTokBytes + 127) / 128 * 128;
    static constexpr int kRowVecs = KDA ? 4 : 3;
    static constexpr int kBlock = 16;
    // per tile slot: row vectors; per warp (two): -s and 1/s of the block's rows for its two groups
    static constexpr int kWarpScratch = 4 * kBlock * 4;
    static constexpr int kSlotBytes = (kRowVecs * D * 4 + 2 * kWarpScratch + 127) / 128 * 128;
    static constexpr int kHeader = 256;
};

template <int D, int KH, bool KDA, typename TI, typename TO, bool FUSED>
__global__ void __launch_bounds__(512, 1) damp_decode_kernel(const __grid_constant__ StepParamsDamp P) {
    using S = DampShape<D, KH, KDA, TI>;
    constexpr int WPT = 2;
    constexpr int NG = S::kGroups;
    static_assert(D == 128 && NG == 4, "two warps of 64 columns, groups of 32");
    static_assert((D - KH) % S::kBlock == 0 && KH % 4 == 0, "INT8 rows fill whole blocks");

    extern __shared__ __align__(128) uint8_t smem[];
    const int W = blockDim.x >> 5;
    const int NSLOT = W / WPT;
    const int w = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ps = w / WPT;
    const int wt = w - ps * WPT;
    const int tt = wt * 32 + lane;
    const int cA = 64 * wt + lane, cB = cA + 32;  // this lane's columns: groups 2wt and 2wt + 1
    const int NS = P.stages;
    const int Hv = P.Hv, Hk = P.Hk;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    volatile int32_t *useq = reinterpret_cast<volatile int32_t *>(smem + 128);
    uint8_t *pi_s = smem + S::kHeader;
    float *wv = reinterpret_cast<float *>(smem + P.header_bytes + (size_t)ps * S::kSlotBytes);
    float *nsc = wv + S::kRowVecs * D + wt * 4 * S::kBlock;  // [-sA | -sB | 1/sA | 1/sB] x kBlock
    uint8_t *stages = smem + P.header_bytes + (size_t)NSLOT * S::kSlotBytes;

    if (threadIdx.x < NS) {
        mbar_init(&bars[threadIdx.x], 1);
        useq[threadIdx.x] = -1;
    }
    for (int i = threadIdx.x; i < Hv * D; i += blockDim.x) pi_s[i] = P.pi[i];
    fence_mbar_init();
    pdl_launch_next();
    pdl_wait();  // the previous kernel's writes are visible from here on
    __syncthreads();

    auto tile_sync = [&]() { group_sync(1 + ps, 32 * WPT); };

    const int items = P.B * Hv;
    const int grid = gridDim.x;
    const TI *q_g = static_cast<const TI *>(P.q);
    const TI *k_g = static_cast<const TI *>(P.k);
    const TI *v_g = static_cast<const TI *>(P.v);
    uint8_t *pool = static_cast<uint8_t *>(P.pool);
    auto item_of = [&](int j) -> int { return (int)blockIdx.x + j * grid; };
    auto slot_ok = [&](int32_t s) { return s >= 0 && (int64_t)s < P.n_slots; };

    auto issue = [&](int j) {
        const int it = item_of(j);
        if (it >= items) return;
        const int s = j % NS;
        uint64_t *bar = &bars[s];
        uint8_t *st = stages + (size_t)s * S::kStage;
        const int b = it / Hv, h = it - b * Hv;
        const int g = h / (Hv / Hk);
        const int32_t slot = P.slot_idx[b];
        useq[s] = j / NS;
        if (!slot_ok(slot)) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, (uint32_t)(S::kStateBytes + S::kTokBytes));
        bulk_g2s(st, pool + ((size_t)slot * Hv + h) * S::kStateBytes, S::kStateBytes, bar);
        uint8_t *tb = st + S::kStatePad;
        bulk_g2s(tb, k_g + ((size_t)b * Hk + g) * D, S::kVecBytes, bar);
        bulk_g2s(tb + S::kVecBytes, q_g + ((size_t)b * Hk + g) * D, S::kVecBytes, bar);
        bulk_g2s(tb + 2 * S::kVecBytes, v_g + ((size_t)b * Hv + h) * D, S::kVecBytes, bar);
        if (KDA) bulk_g2s(tb + 3 * S::kVecBytes, P.alpha + ((size_t)b * Hv + h) * D, D * 4, bar);
    };

    if (threadIdx.x == 0)
        for (int j = 0; j < NS; ++j) issue(j);

    auto tile_beta = [&](int it) -> float { return it < items ? P.beta[it] : 0.0f; };
    auto tile_alpha = [&](int it) -> float { return (!KDA && it < items) ? P.alpha[it] : 0.0f; };
    // pool slot of a tile (for its stores), read one tile ahead too
    auto tile_slot = [&](int it) -> int32_t { return it < items ? P.slot_idx[it / Hv] : -1; };
    float nbeta = tile_beta(item_of(ps)), nalpha = tile_alpha(item_of(ps));
    int32_t nslot = tile_slot(item_of(ps));
    const bool l0 = lane & 1, l1 = lane & 2, l2 = lane & 4, l3 = lane & 8;

    for (int j = ps;; j += NSLOT) {
        const int it = item_of(j);
        if (it >= items) break;
        const float beta0 = nbeta, alpha0 = nalpha;
        const int32_t slot = nslot;
        nbeta = tile_beta(item_of(j + NSLOT));
        nalpha = tile_alpha(item_of(j + NSLOT));
        nslot = tile_slot(item_of(j + NSLOT));
        const int s = j % NS;
        const int32_t use = j / NS;

        bool ok = false;
        for (uint32_t n = 0; n < kWaitPollLimit; ++n) {
            if (useq[s] == use) {
                ok = true;
                break;
            }
            __nanosleep(64);
        }
        ok = ok && (mbar_wait_bounded(&bars[s], (uint32_t)use & 1u) ||
                    mbar_wait_bounded(&bars[s], (uint32_t)use & 1u));
        if (group_sync_or(1 + ps, 32 * WPT, !ok)) {
            if (tt == 0) report(P.status, 8);
            return;
        }
        const int b = it / Hv, h = it - b * Hv;
        if (!slot_ok(slot)) {
            if (tt == 0) {
                report(P.status, 1);
                issue(j + NS);
            }
            __syncwarp();
            continue;
        }
        uint8_t *st = stages + (size_t)s * S::kStage;
        const uint8_t *tb = st + S::kStatePad;

        // ---- row vectors: thread tt builds rows 2tt, 2tt + 1 ----------------
        {
            const uint32_t srcs = *reinterpret_cast<const uint16_t *>(pi_s + h * D + 2 * tt);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int src = (srcs >> (8 * i)) & 0xff;
                const float kf = load_as_f32<TI>(reinterpret_cast<const TI *>(tb) + src);
                wv[2 * tt + i] = kf;
                wv[D + 2 * tt + i] = __fmul_rn(beta0, kf);
                wv[2 * D + 2 * tt + i] = load_as_f32<TI>(reinterpret_cast<const TI *>(tb + S::kVecBytes) + src);
                const float ar = KDA ? reinterpret_cast<const float *>(tb + 3 * S::kVecBytes)[src] : alpha0;
                if (KDA) wv[3 * D + 2 * tt + i] = ar;
            }
        }
        // value-scaling factors of this lane's columns; v' = v / c'
        const float csA = P.cs[h * D + cA], csB = P.cs[h * D + cB];
        const float vA = __fdiv_rn(load_as_f32<TI>(reinterpret_cast<const TI *>(tb + 2 * S::kVecBytes) + cA), csA);
        const float vB = __fdiv_rn(load_as_f32<TI>(reinterpret_cast<const TI *>(tb + 2 * S::kVecBytes) + cB), csB);
        tile_sync();

        const float4 *K4 = reinterpret_cast<const float4 *>(wv);
        const float4 *BK4 = reinterpret_cast<const float4 *>(wv + D);
        const float4 *Q4 = reinterpret_cast<const float4 *>(wv + 2 * D);
        const float4 *A4 = reinterpret_cast<const float4 *>(wv + 3 * D);
        uint32_t *hiw = reinterpret_cast<uint32_t *>(st);               // FP16 pairs [KH/2][D]
        uint32_t *low = reinterpret_cast<uint32_t *>(st + 2 * KH * D);  // INT8 quads [(D-KH)/4][D]
        float *scales = reinterpret_cast<float *>(st + 2 * KH * D + (D - KH) * D);  // [(D-KH)][NG]
        uint8_t *dst = pool + ((size_t)slot * Hv + h) * S::kStateBytes;  // the tile in HBM
        uint32_t *hi_g = reinterpret_cast<uint32_t *>(dst);
        uint32_t *lo_g = reinterpret_cast<uint32_t *>(dst + 2 * KH * D);
        float *scales_g = reinterpret_cast<float *>(dst + 2 * KH * D + (D - KH) * D);
        // this lane's column cA in each region (column cB is 32 words further);
        // the warp's two group scales of a row are a float2 at 2 wt
        const uint32_t *hiA = hiw + cA, *lowA = low + cA;
        uint32_t *hiA_g = hi_g + cA, *loA_g = lo_g + cA;
        const float *scW = scales + 2 * wt;

        // x[i] = columns (cA, cB) of row 4q + i
        auto decay = [&](int q, float2 (&x)[4]) {
            const float4 a = KDA ? A4[q] : make_float4(alpha0, alpha0, alpha0, alpha0);
            const float ar[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = __fmul2_rn(x[i], make_float2(ar[i], ar[i]));
        };
        auto load_hi = [&](int q, float2 (&x)[4]) {
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const uint32_t wa = hiA[(2 * q + pr) * D], wb = hiA[(2 * q + pr) * D + 32];
                const __half2 ha = *reinterpret_cast<const __half2 *>(&wa);
                const __half2 hb = *reinterpret_cast<const __half2 *>(&wb);
                x[2 * pr] = make_float2(__low2float(ha), __low2float(hb));
                x[2 * pr + 1] = make_float2(__high2float(ha), __high2float(hb));
            }
            decay(q, x);
        };
        auto load_lo = [&](int qd, float2 (&x)[4]) {
            const uint32_t *lw = lowA + qd * D;
            const uint32_t wa = lw[0] ^ 0x80808080u, wb = lw[32] ^ 0x80808080u;
            const float *sq = scW + 4 * qd * NG;
            const float2 nb = make_float2(-kCodeBias, -kCodeBias);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 s2 = *reinterpret_cast<const float2 *>(sq + i * NG);
                const uint32_t sel = 0x7540u + (uint32_t)i;
                const float fa = __uint_as_float(__byte_perm(wa, 0x4B000000u, sel));
                const float fb = __uint_as_float(__byte_perm(wb, 0x4B000000u, sel));
                x[i] = __fmul2_rn(__fadd2_rn(make_float2(fa, fb), nb), s2);
            }
            decay(KH / 4 + qd, x);
        };
        auto predict = [&](int q, const float2 (&x)[4], float2 &p) {
            const float4 k4 = K4[q];
            const float kr[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) p = __ffma2_rn(x[i], make_float2(kr[i], kr[i]), p);
        };
        auto write_read = [&](int q, float2 (&x)[4], float2 e, float2 &o) {
            const float4 b4 = BK4[q];
            const float4 q4 = Q4[q];
            const float br[4] = {b4.x, b4.y, b4.z, b4.w};
            const float qr[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[i] = __ffma2_rn(make_float2(br[i], br[i]), e, x[i]);
                o = __ffma2_rn(x[i], make_float2(qr[i], qr[i]), o);
            }
        };

        // ---- pass 1: decay and prediction ------------------------------------
        float2 p = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < KH / 4; ++q) {
            float2 x[4];
            load_hi(q, x);
            predict(q, x, p);
        }
#pragma unroll 4
        for (int qd = 0; qd < (D - KH) / 4; ++qd) {
            float2 x[4];
            load_lo(qd, x);
            predict(KH / 4 + qd, x, p);
        }
        const float2 e = make_float2(__fsub_rn(vA, p.x), __fsub_rn(vB, p.y));

        // ---- pass 2: write, readout, requantise ------------------------------
        float2 o = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < KH / 4; ++q) {
            float2 x[4];
            load_hi(q, x);
            write_read(q, x, e, o);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const __half2 ha = __floats2half2_rn(x[2 * pr].x, x[2 * pr + 1].x);
                const __half2 hb = __floats2half2_rn(x[2 * pr].y, x[2 * pr + 1].y);
                hiA_g[(2 * q + pr) * D] = *reinterpret_cast<const uint32_t *>(&ha);
                hiA_g[(2 * q + pr) * D + 32] = *reinterpret_cast<const uint32_t *>(&hb);
            }
        }
        constexpr int QB = S::kBlock / 4;
#pragma unroll 1
        for (int blk = 0; blk < (D - KH) / S::kBlock; ++blk) {
            const int q0 = blk * QB;
            float2 X[QB][4];
#pragma unroll
            for (int qq = 0; qq < QB; ++qq) {
                load_lo(q0 + qq, X[qq]);
                write_read(KH / 4 + q0 + qq, X[qq], e, o);
            }
            // group maxima: one warp max-reduction per (row, group)
            float ra[S::kBlock], rb[S::kBlock];
#pragma unroll
            for (int qq = 0; qq < QB; ++qq)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ra[4 * qq + i] = warp_max_abs_nan(X[qq][i].x);
                    rb[4 * qq + i] = warp_max_abs_nan(X[qq][i].y);
                }
            auto pick = [&](const float (&r)[S::kBlock]) {  // lane i (and i + 16) gets r[i]
                float t8[8], t4[4], t2[2];
#pragma unroll
                for (int i = 0; i < 8; ++i) t8[i] = l0 ? r[2 * i + 1] : r[2 * i];
#pragma unroll
                for (int i = 0; i < 4; ++i) t4[i] = l1 ? t8[2 * i + 1] : t8[2 * i];
#pragma unroll
                for (int i = 0; i < 2; ++i) t2[i] = l2 ? t4[2 * i + 1] : t4[2 * i];
                return l3 ? t2[1] : t2[0];
            };
            const float ma = pick(ra), mb = pick(rb);
            bool nonfinite = false;
            if (lane < S::kBlock) {
                const float sa = row_scale_from_absmax(ma), sb = row_scale_from_absmax(mb);
                nsc[lane] = -sa;
                nsc[S::kBlock + lane] = -sb;
                const bool bad_a = !(ma <= 3.402823466e38f), bad_b = !(mb <= 3.402823466e38f);
                // fused arithmetic: y = 0 marks a group whose absmax is inf or NaN
                nsc[2 * S::kBlock + lane] = (FUSED && bad_a) ? 0.0f : __frcp_rn(sa);
                nsc[3 * S::kBlock + lane] = (FUSED && bad_b) ? 0.0f : __frcp_rn(sb);
                *reinterpret_cast<float2 *>(scales_g + (blk * S::kBlock + lane) * NG + 2 * wt) = make_float2(sa, sb);
                nonfinite = bad_a || bad_b;
            }
            __syncwarp();
            nonfinite = __any_sync(0xffffffffu, nonfinite);
            if (!nonfinite) {
#pragma unroll
                for (int qq = 0; qq < QB; ++qq) {
                    const float4 na4 = reinterpret_cast<const float4 *>(nsc)[qq];
                    const float4 nb4 = reinterpret_cast<const float4 *>(nsc + S::kBlock)[qq];
                    const float4 ya4 = reinterpret_cast<const float4 *>(nsc + 2 * S::kBlock)[qq];
                    const float4 yb4 = reinterpret_cast<const float4 *>(nsc + 3 * S::kBlock)[qq];
                    const float na[4] = {na4.x, na4.y, na4.z, na4.w}, nbv[4] = {nb4.x, nb4.y, nb4.z, nb4.w};
                    const float ya[4] = {ya4.x, ya4.y, ya4.z, ya4.w}, yb[4] = {yb4.x, yb4.y, yb4.z, yb4.w};
                    uint32_t mA[4], mB[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 x = X[qq][i];
                        const float2 y = make_float2(ya[i], yb[i]);
                        float2 t;
                        if constexpr (FUSED) {  // integer nearest to x y, rounded once
                            t = __ffma2_rn(x, y, make_float2(kRound, kRound));
                        } else {                // RN(x / s), then rounded to an integer
                            const float2 n = make_float2(na[i], nbv[i]);
                            t = __fmul2_rn(x, y);
                            t = __ffma2_rn(__ffma2_rn(t, n, x), y, t);
                            t = __ffma2_rn(__ffma2_rn(t, n, x), y, t);
                            t = __fadd2_rn(t, make_float2(kRound, kRound));
                        }
                        mA[i] = __float_as_uint(t.x);
                        mB[i] = __float_as_uint(t.y);
                    }
                    uint32_t *lg = loA_g + (q0 + qq) * D;
                    lg[0] = __byte_perm(__byte_perm(mA[0], mA[1], 0x0040), __byte_perm(mA[2], mA[3], 0x0040), 0x5410);
                    lg[32] = __byte_perm(__byte_perm(mB[0], mB[1], 0x0040), __byte_perm(mB[2], mB[3], 0x0040), 0x5410);
                }
            } else {
#pragma unroll
                for (int qq = 0; qq < QB; ++qq) {
                    uint32_t wa = 0, wb = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float s_a = -nsc[4 * qq + i], s_b = -nsc[S::kBlock + 4 * qq + i];
                        if constexpr (FUSED) {
                            wa |= quant_rcp_or_exact(X[qq][i].x, s_a, nsc[2 * S::kBlock + 4 * qq + i]) << (8 * i);
                            wb |= quant_rcp_or_exact(X[qq][i].y, s_b, nsc[3 * S::kBlock + 4 * qq + i]) << (8 * i);
                        } else {
                            wa |= quant_exact(X[qq][i].x, s_a) << (8 * i);
                            wb |= quant_exact(X[qq][i].y, s_b) << (8 * i);
                        }
                    }
                    loA_g[(q0 + qq) * D] = wa;
                    loA_g[(q0 + qq) * D + 32] = wb;
                }
            }
            __syncwarp();
        }
        if (P.o) {
            TO *og = static_cast<TO *>(P.o) + ((size_t)b * Hv + h) * D;
            store_from_f32<TO>(og + cA, __fmul_rn(csA, o.x));
            store_from_f32<TO>(og + cB, __fmul_rn(csB, o.y));
        }

        // the stage has been read by both warps: it takes tile j + NS
        tile_sync();
        if (tt == 0) {
            fence_proxy_async_smem();
            issue(j + NS);
        }
        __syncwarp();
    }
}

}  // namespace rs
