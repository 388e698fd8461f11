// rs_prefill.cuh -- prefill chunks on the state pool (sm_103a): the kernel and
// its dispatch, instantiated per layout family in rs_prefill.cu (FP32),
// rs_prefill_mixed.cu and rs_prefill_damp.cu.
//
// DAMP Appendix A.4 "Prefill path": prefill runs FP32 arithmetic within each
// chunk and writes its final state to the same packed cache, which later
// chunks and decoding steps read.  One group of D threads advances one state
// tile (sequence b, value head h) through the n_b tokens of its chunk: the
// tile is read (and, for the mixed layout, dequantised) once into registers,
// thread v owning column v as row pairs, each token is one decode step on the
// registers (decay, prediction p = S^T k, error, rank-1 write, readout
// o = S^T q, with both sums sequential in ascending physical row order), and
// the tile is written (requantised) once.  The result therefore equals n_b
// decode steps of the FP32 layout bit for bit, and the multi-token replay of
// the oracle on the mixed layout (one dequantisation, one requantisation).
//
// Token inputs are gathered by the group's threads (thread u reads key
// channel pi[u] of k, q and the decay, and value u of v) one token ahead into
// registers, so their global-load latency hides behind the current token's
// two passes; they reach shared memory as per-row vectors in one of two
// buffers, one group barrier per token.
//
// DAMP-exact layout (GRP: INT8 groups of 32 values along dv, value scaling;
// DAMP Appendix A.1, A.3 Eq. 17-18): thread v's column lies in scale group
// v / 32, which is the thread's warp, so a group's row maximum is one warp
// max-reduction; the value v is divided by the column's factor c'_v before
// the error and the readout is multiplied by it.  Multi-token replay on that
// layout runs through this kernel too (it computes the same thing).
#pragma once

#include "rs_damp.h"
#include "rs_quant.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

// Shared memory of one group: row vectors [2 buffers][NV][D] floats, then the
// requantisation scratch of the mixed layout (partial maxima [D/32][D], row
// scales, their negations and reciprocals [D] each, a flag word); the
// requantised words go from registers straight to the pool tile.
template <int D, int KHI, bool KDA, bool GRP>
struct PrefillShape {
    static constexpr bool kMixed = KHI >= 0;
    static constexpr int kKhi = KHI < 0 ? 0 : KHI;
    static constexpr int kNV = KDA ? 5 : 4;  // K, BK, Q, V (+ A)
    static constexpr int kScales = GRP ? D / kDampGroup : 1;  // INT8 scales per row
    static constexpr int kStateBytes =
        kMixed ? (2 * kKhi * D + (D - kKhi) * D + 4 * (D - kKhi) * kScales) : D * D * 4;
    static constexpr int kRowBytes = 2 * kNV * D * 4;
    static constexpr int kScratch = kMixed ? ((D / 32) * D * 4 + 3 * D * 4 + 128) : 0;
    static constexpr int kRegion = (kRowBytes + kScratch + 127) / 128 * 128;
};

// DAMP-exact tile: dequantise column tid (group tid / 32) into row pairs;
// `scales` ([D - KH][D / 32] floats) replaces the tile's scales when given.
template <int D, int KH>
__device__ __forceinline__ void damp_dequant(const uint8_t *tile, int tid, float2 (&xs)[D / 2],
                                             const float *scales) {
    constexpr int NG = D / kDampGroup;
    const __half2 *hi = reinterpret_cast<const __half2 *>(tile);
    const uint32_t *lo = reinterpret_cast<const uint32_t *>(tile + 2 * KH * D);
    const float *sc = scales ? scales : reinterpret_cast<const float *>(tile + 2 * KH * D + (D - KH) * D);
    const int gi = tid / kDampGroup;
#pragma unroll
    for (int j = 0; j < KH / 2; ++j) xs[j] = __half22float2(hi[j * D + tid]);
#pragma unroll
    for (int qd = 0; qd < (D - KH) / 4; ++qd) {
        const uint32_t w = lo[qd * D + tid] ^ 0x80808080u;
        const float s0 = sc[(4 * qd) * NG + gi], s1 = sc[(4 * qd + 1) * NG + gi];
        const float s2 = sc[(4 * qd + 2) * NG + gi], s3 = sc[(4 * qd + 3) * NG + gi];
        const float f0 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540));
        const float f1 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541));
        const float f2 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542));
        const float f3 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543));
        const float2 c01 = __fadd2_rn(make_float2(f0, f1), make_float2(-kCodeBias, -kCodeBias));
        const float2 c23 = __fadd2_rn(make_float2(f2, f3), make_float2(-kCodeBias, -kCodeBias));
        xs[KH / 2 + 2 * qd] = __fmul2_rn(c01, make_float2(s0, s1));
        xs[KH / 2 + 2 * qd + 1] = __fmul2_rn(c23, make_float2(s2, s3));
    }
}

// DAMP-exact tile: requantise column tid from its row pairs into `out`
// (shared memory, the tile's byte layout).  The group of column tid is the
// thread's warp: a row's group maximum is one warp max-reduction; every lane
// forms the same scale, lane 0 stores it.  Codes: the IEEE quotient, or the
// fused arithmetic's one-rounding product (groups with a non-finite maximum
// keep the quotient).
template <int D, int KH, bool FUSED>
__device__ __forceinline__ void damp_requant(const float2 (&xs)[D / 2], uint8_t *out, int tid, int lane) {
    constexpr int NG = D / kDampGroup;
    __half2 *hi = reinterpret_cast<__half2 *>(out);
    uint32_t *lo = reinterpret_cast<uint32_t *>(out + 2 * KH * D);
    float *sc = reinterpret_cast<float *>(out + 2 * KH * D + (D - KH) * D);
    const int gi = tid / kDampGroup;
#pragma unroll
    for (int j = 0; j < KH / 2; ++j) hi[j * D + tid] = __floats2half2_rn(xs[j].x, xs[j].y);
#pragma unroll
    for (int qd = 0; qd < (D - KH) / 4; ++qd) {
        const float xr[4] = {xs[KH / 2 + 2 * qd].x, xs[KH / 2 + 2 * qd].y, xs[KH / 2 + 2 * qd + 1].x,
                             xs[KH / 2 + 2 * qd + 1].y};
        uint32_t word = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = warp_max_abs_nan(xr[i]);
            const float sv = row_scale_from_absmax(a);
            uint32_t c;
            if constexpr (FUSED) c = quant_rcp_or_exact(xr[i], sv, a <= 3.402823466e38f ? __frcp_rn(sv) : 0.0f);
            else c = quant_exact(xr[i], sv);
            word |= c << (8 * i);
            if (lane == 0) sc[(4 * qd + i) * NG + gi] = sv;
        }
        lo[qd * D + tid] = word;
    }
}

// Threads per CTA: three groups for the FP32 layout (its requantisation-free
// code fits the 170 registers that allows), two for the mixed layouts.
constexpr int prefill_threads(int khi) { return khi < 0 ? 384 : 256; }

template <int D, int KHI, bool KDA, typename TI, typename TO, bool FUSED, bool GRP, typename PT>
__global__ void __launch_bounds__(prefill_threads(KHI), 1) prefill_kernel(const __grid_constant__ PT P) {
    using S = PrefillShape<D, KHI, KDA, GRP>;
    constexpr bool MIXED = S::kMixed;
    constexpr int KH = S::kKhi;
    constexpr int DP = D / 2;
    constexpr int NV = S::kNV;

    extern __shared__ __align__(128) uint8_t smem[];
    const int G = blockDim.x / D;
    const int grp = threadIdx.x / D;
    const int tid = threadIdx.x - grp * D;
    const int lane = threadIdx.x & 31;
    const int wig = tid >> 5;
    const uint32_t bar_id = 1 + grp;
    uint8_t *region = smem + (size_t)grp * S::kRegion;
    float *rowv = reinterpret_cast<float *>(region);  // [2][NV][D]
    float *red = rowv + 2 * NV * D;                    // mixed: [D/32][D]
    float *scl = red + (D / 32) * D;
    float *nscl = scl + D;
    float *rcp = nscl + D;
    int *flag = reinterpret_cast<int *>(rcp + D);

    const int Hv = P.Hv, Hk = P.Hk, L = P.L;
    const int items = P.B * Hv;
    const TI *q_g = static_cast<const TI *>(P.q);
    const TI *k_g = static_cast<const TI *>(P.k);
    const TI *v_g = static_cast<const TI *>(P.v);
    TO *og = static_cast<TO *>(P.o);
    pdl_launch_next();
    pdl_wait();  // the previous kernel's writes are visible from here on

    for (int item = blockIdx.x * G + grp; item < items; item += gridDim.x * G) {
        const int b = item / Hv, h = item - (item / Hv) * Hv;
        const int g = h / (Hv / Hk);
        const int32_t slot = P.slot_idx[b];
        const int32_t n = P.n_tokens ? P.n_tokens[b] : L;
        // every thread of the group sees the same item: the skips are uniform
        if (slot < 0 || (int64_t)slot >= P.n_slots) {
            if (tid == 0) report(P.status, 1);
            continue;
        }
        if (n < 0 || n > L) {
            if (tid == 0) report(P.status, 2);
            continue;
        }
        if (n == 0) continue;
        const int src = MIXED ? (int)P.pi[h * D + tid] : tid;  // key channel of physical row tid
        float csv = 1.0f;  // DAMP-exact: the value-scaling factor c'_v of column tid
        if constexpr (GRP) csv = P.cs[h * D + tid];

        // inputs of token t for row tid (key channel src) and value tid
        auto load_tok = [&](int t, float &kf, float &qf, float &vf, float &af, float &bt) {
            const size_t bl = (size_t)b * L + t;
            kf = load_as_f32<TI>(k_g + (bl * Hk + g) * D + src);
            qf = load_as_f32<TI>(q_g + (bl * Hk + g) * D + src);
            vf = load_as_f32<TI>(v_g + (bl * Hv + h) * D + tid);
            af = KDA ? P.alpha[(bl * Hv + h) * D + src] : P.alpha[bl * Hv + h];
            bt = P.beta[bl * Hv + h];
        };
        auto put_tok = [&](int buf, float kf, float qf, float vf, float af, float bt) {
            float *rv = rowv + buf * NV * D;
            rv[tid] = kf;
            rv[D + tid] = __fmul_rn(bt, kf);
            rv[2 * D + tid] = qf;
            rv[3 * D + tid] = GRP ? __fdiv_rn(vf, csv) : vf;  // DAMP-exact: v' = v / c'
            if (KDA) rv[4 * D + tid] = af;
        };

        float kf, qf, vf, af, bt;
        load_tok(0, kf, qf, vf, af, bt);
        put_tok(0, kf, qf, vf, af, bt);
        float a_cur = af;  // GDN: the scalar decay of the current token
        group_sync(bar_id, D);  // token 0's row vectors visible

        // ---- the tile -> registers (dequantised once) ---------------------
        float2 x[DP];
        const size_t tile_off = ((size_t)slot * Hv + h) * S::kStateBytes;
        const uint8_t *tile = static_cast<const uint8_t *>(P.pool) + tile_off;
        if constexpr (!MIXED) {
            const float *st = reinterpret_cast<const float *>(tile);
#pragma unroll
            for (int j = 0; j < DP; ++j) x[j] = make_float2(st[(2 * j) * D + tid], st[(2 * j + 1) * D + tid]);
        } else if constexpr (GRP) {
            damp_dequant<D, KH>(tile, tid, x, nullptr);
        } else {
            mixed_dequant<D, KH>(tile, tid, x);
        }

        // ---- the chunk's tokens --------------------------------------------
        for (int t = 0; t < n; ++t) {
            const float *rv = rowv + (t & 1) * NV * D;
            const bool more = t + 1 < n;
            float kn = 0.0f, qn = 0.0f, vn = 0.0f, an = 0.0f, bn = 0.0f;
            if (more) load_tok(t + 1, kn, qn, vn, an, bn);  // latency hidden by the passes below

            float p = 0.0f;
#pragma unroll
            for (int j = 0; j < DP; j += 2) {
                const float4 kk = *reinterpret_cast<const float4 *>(rv + 2 * j);
                float4 aa;
                if (KDA) aa = *reinterpret_cast<const float4 *>(rv + 4 * D + 2 * j);
                else aa = make_float4(a_cur, a_cur, a_cur, a_cur);
                x[j] = __fmul2_rn(x[j], make_float2(aa.x, aa.y));
                x[j + 1] = __fmul2_rn(x[j + 1], make_float2(aa.z, aa.w));
                p = __fmaf_rn(x[j].x, kk.x, p);
                p = __fmaf_rn(x[j].y, kk.y, p);
                p = __fmaf_rn(x[j + 1].x, kk.z, p);
                p = __fmaf_rn(x[j + 1].y, kk.w, p);
            }
            const float e = __fsub_rn(rv[3 * D + tid], p);
            float o = 0.0f;
#pragma unroll
            for (int j = 0; j < DP; j += 2) {
                const float4 bk = *reinterpret_cast<const float4 *>(rv + D + 2 * j);
                const float4 qq = *reinterpret_cast<const float4 *>(rv + 2 * D + 2 * j);
                x[j] = __ffma2_rn(make_float2(bk.x, bk.y), make_float2(e, e), x[j]);
                x[j + 1] = __ffma2_rn(make_float2(bk.z, bk.w), make_float2(e, e), x[j + 1]);
                o = __fmaf_rn(x[j].x, qq.x, o);
                o = __fmaf_rn(x[j].y, qq.y, o);
                o = __fmaf_rn(x[j + 1].x, qq.z, o);
                o = __fmaf_rn(x[j + 1].y, qq.w, o);
            }
            if (og) store_from_f32<TO>(og + (((size_t)b * L + t) * Hv + h) * D + tid, GRP ? __fmul_rn(csv, o) : o);
            if (more) {
                // buffer (t + 1) & 1 was last read by token t - 1, finished
                // before the previous barrier
                put_tok((t + 1) & 1, kn, qn, vn, an, bn);
                a_cur = an;
            }
            group_sync(bar_id, D);  // token t + 1's row vectors visible
        }

        // ---- registers -> the pool (requantised once) -----------------------
        uint8_t *dst = static_cast<uint8_t *>(P.pool) + tile_off;
        if constexpr (!MIXED) {
            float *st = reinterpret_cast<float *>(dst);
#pragma unroll
            for (int j = 0; j < DP; ++j) {
                st[(2 * j) * D + tid] = x[j].x;
                st[(2 * j + 1) * D + tid] = x[j].y;
            }
        } else if constexpr (GRP) {
            // the requantised words go from registers straight to the pool tile
            damp_requant<D, KH, FUSED>(x, dst, tid, lane);
        } else {
            float mine[D / 32];
#pragma unroll
            for (int k = 0; k < D / 32; ++k) mine[k] = 0.0f;
#pragma unroll
            for (int j = KH / 2; j < DP; ++j) absmax_pair<D>(x[j], j, lane, mine);
            mixed_requant_from_max<D, KH, FUSED>(x, mine, dst, red, scl, nscl, rcp, flag, tid, lane, wig,
                                                 bar_id, [&] {
                                                     if (tid == 0) *flag = 0;
                                                 });
        }
        group_sync(bar_id, D);  // row vectors and scratch free for the next item
    }
}

template <int D, int KHI, bool KDA, typename TI, typename TO, bool FUSED, bool GRP, typename PT>
cudaError_t run(PT &P, cudaStream_t s) {
    using Sh = PrefillShape<D, KHI, KDA, GRP>;
    auto kern = prefill_kernel<D, KHI, KDA, TI, TO, FUSED, GRP, PT>;
    constexpr int G = prefill_threads(KHI) / D;
    const int smem = G * Sh::kRegion;
    const int groups_needed = (P.B * P.Hv + G - 1) / G;
    int grid = device_sm_count();
    if (grid > groups_needed) grid = groups_needed;
    if (grid < 1) grid = 1;
    cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(G * D), smem, s, P);
}

template <int D, int KHI, bool KDA, bool FUSED, bool GRP, typename PT>
cudaError_t by_types(const StepLaunch &L, PT &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32)
        return run<D, KHI, KDA, __nv_bfloat16, float, FUSED, GRP>(P, s);
    if (L.in_dt == RS_BF16 && L.out_dt == RS_BF16)
        return run<D, KHI, KDA, __nv_bfloat16, __nv_bfloat16, FUSED, GRP>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<D, KHI, KDA, float, float, FUSED, GRP>(P, s);
    if (L.in_dt == RS_F16 && L.out_dt == RS_F32) return run<D, KHI, KDA, __half, float, FUSED, GRP>(P, s);
    return cudaErrorNotSupported;
}

template <bool GRP, typename PT>
cudaError_t by_mode(const StepLaunch &L, PT &P, cudaStream_t s) {
    if (L.fused) return L.kda ? by_types<128, 16, true, true, GRP>(L, P, s) : by_types<128, 16, false, true, GRP>(L, P, s);
    return L.kda ? by_types<128, 16, true, false, GRP>(L, P, s) : by_types<128, 16, false, false, GRP>(L, P, s);
}

}  // namespace

// Mixed FP16/INT8 layout (dk = 128, 16 FP16 rows), in rs_prefill_mixed.cu.
cudaError_t launch_prefill_mixed(const StepLaunch &L, PrefillParams &P, cudaStream_t s);

}  // namespace rs
