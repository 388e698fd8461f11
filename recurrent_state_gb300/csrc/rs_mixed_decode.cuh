// rs_mixed_decode.cuh -- single-token decode on the mixed FP16/INT8 layout
// (DAMP §5.2 and Appendix A.4: one fused load, dequantise, update, readout,
// requantise and store per step), one warp per state tile.
//
// Lane l of a warp owns the four adjacent columns 4l..4l+3 of the tile, so
//   * one 16-byte shared load brings a column quad of a word row (4 INT8 rows
//     or 2 FP16 rows per column), and every per-element operation runs as a
//     paired FP32 instruction (mul/add/fma .f32x2) over two columns of one
//     row -- including the two reductions over key channels, which stay
//     sequential ascending-row FMA chains per column, exactly the oracle's
//     evaluation order;
//   * the per-row absmax of the requantisation is a max over the lane's four
//     values plus one warp max-reduction (redux.sync): no shared-memory
//     combine and no barrier beyond the warp.
// The packed tile (18,880 B at d = 128) is worked on in place in its
// shared-memory stage: pass 1 dequantises and decays each row and runs the
// prediction chain p = S^T k; pass 2 repeats the dequantisation and decay
// from the same operands (so they round the same way), applies the write
// x += RN(beta k) e^T, runs the readout chain o = S^T q, and requantises in
// blocks of 16 rows (FP16 rows round to nearest even; INT8 rows get a new
// scale from the block's absmax and an exact RN(x/s) code, as in
// rs_step.cuh).  Lane 0 then bulk-stores the tile.
//
// A CTA runs W warps over a ring of NS > W stages.  Its tiles are numbered
// j = 0, 1, ... (tile blockIdx.x + j * gridDim.x of the launch); tile j uses
// stage j mod NS and warp j mod W.  The warp that finishes tile j issues the
// bulk copy of tile j + NS into the stage it has just released, so the copy
// of a tile starts NS - W tiles ahead of the warp that takes it.  A use
// counter per stage, written before each copy is issued, tells a warp that
// its copy was issued before it waits on the stage's mbarrier parity (tiles
// are taken by different warps, so the parity alone could alias).  Every wait
// is bounded and reports RS_DEV_PIPE_TIMEOUT.
#pragma once

#include "rs_step.cuh"

namespace rs {

constexpr int kMixedWarps = 8;       // warps per CTA
constexpr int kMixedMaxStages = 16;  // stage ring length limit (mbarriers in the header)

template <int D, int KH, bool KDA, typename TI>
struct MixedWarpShape {
    static constexpr int kStateBytes = 2 * KH * D + (D - KH) * D + 4 * (D - KH);
    static constexpr int kStatePad = (kStateBytes + 127) / 128 * 128;
    static constexpr int kVecBytes = D * (int)sizeof(TI);
    static constexpr int kTokBytes = 3 * kVecBytes + (KDA ? D * 4 : 0);  // k, q, v (+ alpha)
    static constexpr int kStage = (kStatePad + kTokBytes + 127) / 128 * 128;
    static constexpr int kRowVecs = KDA ? 4 : 3;  // K, BK, Q (+ A), floats in row order
    static constexpr int kBlock = 16;             // rows per requantisation block
    // per warp: row vectors, then -s and 1/s of the current block
    static constexpr int kWarpBytes = (kRowVecs * D * 4 + 2 * kBlock * 4 + 127) / 128 * 128;
    static constexpr int kHeader = 256;  // mbarriers [NS], use counters [NS] at +128
};

// max(|a.x|, |a.y|, |b.x|, |b.y|), NaN when any of them is NaN.
__device__ __forceinline__ float max_abs4_nan(float2 a, float2 b) {
    float r;
    asm("{\n\t.reg .f32 t0, t1;\n\t"
        "max.NaN.f32 t0, %1, %2;\n\t"
        "max.NaN.f32 t1, %3, %4;\n\t"
        "max.NaN.f32 %0, t0, t1;\n\t}"
        : "=f"(r)
        : "f"(fabsf(a.x)), "f"(fabsf(a.y)), "f"(fabsf(b.x)), "f"(fabsf(b.y)));
    return r;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Rows 4q..4q+3 of a lane's columns: x[i][0] = columns (c0, c1) of row
// 4q+i, x[i][1] = columns (c2, c3).
struct Quad {
    float2 x[4][2];
};

template <int D, int KH, bool KDA, typename TI, typename TO>
__global__ void __launch_bounds__(kMixedWarps * 32, 1)
    mixed_decode_kernel(const __grid_constant__ StepParamsPi P) {
    using S = MixedWarpShape<D, KH, KDA, TI>;
    static_assert(D == 128, "four columns per lane");
    static_assert((D - KH) % S::kBlock == 0 && KH % 4 == 0, "INT8 rows fill whole blocks");
    constexpr int NQ = D / 4;  // 16-byte column quads per word row

    extern __shared__ __align__(128) uint8_t smem[];
    const int W = blockDim.x >> 5;
    const int w = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int NS = P.stages;
    const int Hv = P.Hv, Hk = P.Hk;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    volatile int32_t *useq = reinterpret_cast<volatile int32_t *>(smem + 128);
    uint8_t *pi_s = smem + S::kHeader;
    float *wv = reinterpret_cast<float *>(smem + P.header_bytes + (size_t)w * S::kWarpBytes);
    float *nsc = wv + S::kRowVecs * D;  // -s of the block's rows
    float *ysc = nsc + S::kBlock;       // 1/s of the block's rows
    uint8_t *stages = smem + P.header_bytes + (size_t)W * S::kWarpBytes;

    if (threadIdx.x < NS) {
        mbar_init(&bars[threadIdx.x], 1);
        useq[threadIdx.x] = -1;
    }
    for (int i = threadIdx.x; i < Hv * D; i += blockDim.x) pi_s[i] = P.pi[i];
    fence_mbar_init();
    __syncthreads();

    const int items = P.B * Hv;
    const int grid = gridDim.x;
    const TI *q_g = static_cast<const TI *>(P.q);
    const TI *k_g = static_cast<const TI *>(P.k);
    const TI *v_g = static_cast<const TI *>(P.v);
    uint8_t *pool = static_cast<uint8_t *>(P.pool);
    auto item_of = [&](int j) -> int { return (int)blockIdx.x + j * grid; };
    auto slot_ok = [&](int32_t s) { return s >= 0 && (int64_t)s < P.n_slots; };

    // Issue the copy of tile j into stage j mod NS (one thread).  A tile with
    // a bad slot gets no copy; its phase is completed by a plain arrival so
    // that the stage's parity sequence stays in step.
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

    // write strength (and GDN decay) of a tile, read one tile ahead
    auto tile_beta = [&](int it) -> float { return it < items ? P.beta[it] : 0.0f; };
    auto tile_alpha = [&](int it) -> float { return (!KDA && it < items) ? P.alpha[it] : 0.0f; };
    float nbeta = tile_beta(item_of(w)), nalpha = tile_alpha(item_of(w));

    for (int j = w;; j += W) {
        const int it = item_of(j);
        if (it >= items) break;
        const float beta0 = nbeta, alpha0 = nalpha;
        nbeta = tile_beta(item_of(j + W));
        nalpha = tile_alpha(item_of(j + W));
        const int s = j % NS;
        const int32_t use = j / NS;

        // ---- wait until the copy of tile j was issued, then for its bytes --
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
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) {
                report(P.status, 8);
                bulk_store_wait_all();
            }
            return;
        }
        const int b = it / Hv, h = it - b * Hv;
        const int32_t slot = P.slot_idx[b];
        if (!slot_ok(slot)) {
            if (lane == 0) {
                report(P.status, 1);
                issue(j + NS);
            }
            __syncwarp();
            continue;
        }
        uint8_t *st = stages + (size_t)s * S::kStage;
        const uint8_t *tb = st + S::kStatePad;

        // ---- row vectors in physical row order: lane l builds rows 4l..4l+3
        {
            const uint32_t src4 = *reinterpret_cast<const uint32_t *>(pi_s + h * D + 4 * lane);
            float kk[4], bk[4], qq[4], aa[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int src = (src4 >> (8 * i)) & 0xff;
                kk[i] = load_as_f32<TI>(reinterpret_cast<const TI *>(tb) + src);
                bk[i] = __fmul_rn(beta0, kk[i]);
                qq[i] = load_as_f32<TI>(reinterpret_cast<const TI *>(tb + S::kVecBytes) + src);
                aa[i] = KDA ? reinterpret_cast<const float *>(tb + 3 * S::kVecBytes)[src] : 0.0f;
            }
            reinterpret_cast<float4 *>(wv)[lane] = make_float4(kk[0], kk[1], kk[2], kk[3]);
            reinterpret_cast<float4 *>(wv + D)[lane] = make_float4(bk[0], bk[1], bk[2], bk[3]);
            reinterpret_cast<float4 *>(wv + 2 * D)[lane] = make_float4(qq[0], qq[1], qq[2], qq[3]);
            if (KDA) reinterpret_cast<float4 *>(wv + 3 * D)[lane] = make_float4(aa[0], aa[1], aa[2], aa[3]);
        }
        float vv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
            vv[t] = load_as_f32<TI>(reinterpret_cast<const TI *>(tb + 2 * S::kVecBytes) + 4 * lane + t);
        __syncwarp();

        const float4 *K4 = reinterpret_cast<const float4 *>(wv);
        const float4 *BK4 = reinterpret_cast<const float4 *>(wv + D);
        const float4 *Q4 = reinterpret_cast<const float4 *>(wv + 2 * D);
        const float4 *A4 = reinterpret_cast<const float4 *>(wv + 3 * D);
        uint4 *hi4 = reinterpret_cast<uint4 *>(st);               // [KH/2][NQ]
        uint4 *lo4 = reinterpret_cast<uint4 *>(st + 2 * KH * D);  // [(D-KH)/4][NQ]
        float *scales = reinterpret_cast<float *>(st + 2 * KH * D + (D - KH) * D);
        const float4 *sc4 = reinterpret_cast<const float4 *>(scales);

        auto decay = [&](int q, Quad &X) {  // rows 4q..4q+3 times their decay
            const float4 a = KDA ? A4[q] : make_float4(alpha0, alpha0, alpha0, alpha0);
            const float ar[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                X.x[i][0] = __fmul2_rn(X.x[i][0], make_float2(ar[i], ar[i]));
                X.x[i][1] = __fmul2_rn(X.x[i][1], make_float2(ar[i], ar[i]));
            }
        };
        auto load_hi = [&](int q, Quad &X) {  // FP16 rows 4q..4q+3, decayed
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const uint4 hw = hi4[(2 * q + pr) * NQ + lane];
                const __half2 h0 = *reinterpret_cast<const __half2 *>(&hw.x);
                const __half2 h1 = *reinterpret_cast<const __half2 *>(&hw.y);
                const __half2 h2 = *reinterpret_cast<const __half2 *>(&hw.z);
                const __half2 h3 = *reinterpret_cast<const __half2 *>(&hw.w);
                X.x[2 * pr][0] = make_float2(__low2float(h0), __low2float(h1));
                X.x[2 * pr][1] = make_float2(__low2float(h2), __low2float(h3));
                X.x[2 * pr + 1][0] = make_float2(__high2float(h0), __high2float(h1));
                X.x[2 * pr + 1][1] = make_float2(__high2float(h2), __high2float(h3));
            }
            decay(q, X);
        };
        auto load_lo = [&](int qd, Quad &X) {  // INT8 rows KH+4qd .. KH+4qd+3, decayed
            const uint4 wr = lo4[qd * NQ + lane];
            const uint32_t wd[4] = {wr.x ^ 0x80808080u, wr.y ^ 0x80808080u, wr.z ^ 0x80808080u,
                                    wr.w ^ 0x80808080u};
            const float4 s4 = sc4[qd];
            const float sr[4] = {s4.x, s4.y, s4.z, s4.w};
            const float2 nb = make_float2(-kCodeBias, -kCodeBias);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t sel = 0x7540u + (uint32_t)i;
                const float f0 = __uint_as_float(__byte_perm(wd[0], 0x4B000000u, sel));
                const float f1 = __uint_as_float(__byte_perm(wd[1], 0x4B000000u, sel));
                const float f2 = __uint_as_float(__byte_perm(wd[2], 0x4B000000u, sel));
                const float f3 = __uint_as_float(__byte_perm(wd[3], 0x4B000000u, sel));
                X.x[i][0] = __fmul2_rn(__fadd2_rn(make_float2(f0, f1), nb), make_float2(sr[i], sr[i]));
                X.x[i][1] = __fmul2_rn(__fadd2_rn(make_float2(f2, f3), nb), make_float2(sr[i], sr[i]));
            }
            decay(KH / 4 + qd, X);
        };
        auto predict = [&](int q, const Quad &X, float2 &p01, float2 &p23) {
            const float4 k4 = K4[q];
            const float kr[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                p01 = __ffma2_rn(X.x[i][0], make_float2(kr[i], kr[i]), p01);
                p23 = __ffma2_rn(X.x[i][1], make_float2(kr[i], kr[i]), p23);
            }
        };
        auto write_read = [&](int q, Quad &X, float2 e01, float2 e23, float2 &o01, float2 &o23) {
            const float4 b4 = BK4[q];
            const float4 q4 = Q4[q];
            const float br[4] = {b4.x, b4.y, b4.z, b4.w};
            const float qr[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                X.x[i][0] = __ffma2_rn(make_float2(br[i], br[i]), e01, X.x[i][0]);
                X.x[i][1] = __ffma2_rn(make_float2(br[i], br[i]), e23, X.x[i][1]);
                o01 = __ffma2_rn(X.x[i][0], make_float2(qr[i], qr[i]), o01);
                o23 = __ffma2_rn(X.x[i][1], make_float2(qr[i], qr[i]), o23);
            }
        };

        // ---- pass 1: decay and prediction p = S^T k (ascending rows) -------
        float2 p01 = make_float2(0.0f, 0.0f), p23 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < KH / 4; ++q) {
            Quad X;
            load_hi(q, X);
            predict(q, X, p01, p23);
        }
#pragma unroll 4
        for (int qd = 0; qd < (D - KH) / 4; ++qd) {
            Quad X;
            load_lo(qd, X);
            predict(KH / 4 + qd, X, p01, p23);
        }
        const float2 e01 = make_float2(__fsub_rn(vv[0], p01.x), __fsub_rn(vv[1], p01.y));
        const float2 e23 = make_float2(__fsub_rn(vv[2], p23.x), __fsub_rn(vv[3], p23.y));

        // ---- pass 2: write, readout, requantise ---------------------------
        float2 o01 = make_float2(0.0f, 0.0f), o23 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < KH / 4; ++q) {  // FP16 rows: round to nearest even, in place
            Quad X;
            load_hi(q, X);
            write_read(q, X, e01, e23, o01, o23);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const __half2 h0 = __floats2half2_rn(X.x[2 * pr][0].x, X.x[2 * pr + 1][0].x);
                const __half2 h1 = __floats2half2_rn(X.x[2 * pr][0].y, X.x[2 * pr + 1][0].y);
                const __half2 h2 = __floats2half2_rn(X.x[2 * pr][1].x, X.x[2 * pr + 1][1].x);
                const __half2 h3 = __floats2half2_rn(X.x[2 * pr][1].y, X.x[2 * pr + 1][1].y);
                uint4 hw;
                hw.x = *reinterpret_cast<const uint32_t *>(&h0);
                hw.y = *reinterpret_cast<const uint32_t *>(&h1);
                hw.z = *reinterpret_cast<const uint32_t *>(&h2);
                hw.w = *reinterpret_cast<const uint32_t *>(&h3);
                hi4[(2 * q + pr) * NQ + lane] = hw;
            }
        }
        constexpr int QB = S::kBlock / 4;  // quads per block
#pragma unroll 1
        for (int blk = 0; blk < (D - KH) / S::kBlock; ++blk) {  // INT8 rows
            const int q0 = blk * QB;
            Quad X[QB];
#pragma unroll
            for (int qq = 0; qq < QB; ++qq) {
                load_lo(q0 + qq, X[qq]);
                write_read(KH / 4 + q0 + qq, X[qq], e01, e23, o01, o23);
            }
            // per-row absmax over the warp's 128 columns; lane r keeps row r
            float mine = 0.0f;
#pragma unroll
            for (int qq = 0; qq < QB; ++qq)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float r = warp_max_abs_nan(max_abs4_nan(X[qq].x[i][0], X[qq].x[i][1]));
                    mine = lane == 4 * qq + i ? r : mine;
                }
            __syncwarp();  // every lane has read the block's old scales
            bool nonfinite = false;
            if (lane < S::kBlock) {
                const float sv = __fdiv_rn(fmaxf(mine, 1e-8f), 127.0f);
                nsc[lane] = -sv;
                ysc[lane] = __frcp_rn(sv);
                scales[blk * S::kBlock + lane] = sv;
                nonfinite = !(mine <= 3.402823466e38f);  // absmax inf or NaN
            }
            __syncwarp();
            nonfinite = __any_sync(0xffffffffu, nonfinite);
            if (!nonfinite) {
#pragma unroll
                for (int qq = 0; qq < QB; ++qq) {
                    const float4 n4 = reinterpret_cast<const float4 *>(nsc)[qq];
                    const float4 y4 = reinterpret_cast<const float4 *>(ysc)[qq];
                    const float nr[4] = {n4.x, n4.y, n4.z, n4.w};
                    const float yr[4] = {y4.x, y4.y, y4.z, y4.w};
                    uint32_t mb[4][4];  // [row][column]: RN(x/s) + 1.5 * 2^23
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const float2 x = X[qq].x[i][hf];
                            const float2 y = make_float2(yr[i], yr[i]);
                            const float2 n = make_float2(nr[i], nr[i]);
                            float2 t = __fmul2_rn(x, y);
                            t = __ffma2_rn(__ffma2_rn(t, n, x), y, t);
                            t = __ffma2_rn(__ffma2_rn(t, n, x), y, t);
                            t = __fadd2_rn(t, make_float2(kRound, kRound));
                            mb[i][2 * hf] = __float_as_uint(t.x);
                            mb[i][2 * hf + 1] = __float_as_uint(t.y);
                        }
                    }
                    uint32_t wd[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        wd[c] = __byte_perm(__byte_perm(mb[0][c], mb[1][c], 0x0040),
                                            __byte_perm(mb[2][c], mb[3][c], 0x0040), 0x5410);
                    lo4[(q0 + qq) * NQ + lane] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                }
            } else {  // absmax inf or NaN somewhere in the block: literal IEEE division
#pragma unroll
                for (int qq = 0; qq < QB; ++qq) {
                    uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float sv = -nsc[4 * qq + i];
                        wd[0] |= quant_exact(X[qq].x[i][0].x, sv) << (8 * i);
                        wd[1] |= quant_exact(X[qq].x[i][0].y, sv) << (8 * i);
                        wd[2] |= quant_exact(X[qq].x[i][1].x, sv) << (8 * i);
                        wd[3] |= quant_exact(X[qq].x[i][1].y, sv) << (8 * i);
                    }
                    lo4[(q0 + qq) * NQ + lane] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                }
            }
            __syncwarp();  // -s and 1/s are rewritten by the next block
        }
        if (P.o) {
            TO *og = static_cast<TO *>(P.o) + ((size_t)b * Hv + h) * D + 4 * lane;
            store_from_f32<TO>(og, o01.x);
            store_from_f32<TO>(og + 1, o01.y);
            store_from_f32<TO>(og + 2, o23.x);
            store_from_f32<TO>(og + 3, o23.y);
        }

        // ---- store the tile; the stage then takes tile j + NS ---------------
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            bulk_s2g(pool + ((size_t)slot * Hv + h) * S::kStateBytes, st, S::kStateBytes);
            bulk_store_commit();
            bulk_store_wait_read();
            issue(j + NS);
        }
        __syncwarp();
    }
    if (lane == 0) bulk_store_wait_all();
}

}  // namespace rs
