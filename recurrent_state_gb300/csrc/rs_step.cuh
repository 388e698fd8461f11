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
//   * the decay and the rank-1 write are elementwise on registers; the column
//     is held as row pairs so these, and the dequantise / requantise
//     arithmetic of the mixed layout, run as paired FP32 instructions
//     (mul/add/fma .f32x2), two rows per instruction, each lane rounded on
//     its own;
//   * a replay keeps the state on chip across tokens ("Serving recurrent
//     attention", speculative decoding without state snapshots).
// The tile and the token inputs arrive through a 1-D bulk TMA copy
// (cp.async.bulk + mbarrier) into the group's shared-memory stage; as soon as
// the stage has been read into registers the group issues the copy of its
// next tile, so HBM reads of tile i+1 overlap the arithmetic of tile i.
// FP32 tiles go straight from registers to HBM with coalesced stores: 16-byte
// stores for a single token (four lanes transpose a 4 x 4 block by shuffles,
// so a lane writes four consecutive columns of a row), a warp's 32 columns of
// a row for a replay; mixed tiles are requantised from registers into the
// pool tile directly (a thread writes its column of each word row).
//
// Mixed layout (DAMP §5.2, Appendix A.4): FP16 rows and INT8 rows with one
// FP32 scale per row are dequantised into the registers, updated in FP32, and
// requantised in the same pass; the per-row absmax is a warp max-reduction
// (redux.sync) plus a combine over the group's warps in shared memory.  The
// INT8 code is round_half_even(x / s) with x / s the IEEE quotient RN(x/s).
// The kernel forms that quotient without a division: with y = rcp_rn(s)
// (correctly rounded), q0 = RN(x*y), r0 = RN(x - q0*s), q1 = RN(q0 + r0*y)
// is a faithful quotient, and one more correction r1 = RN(x - q1*s),
// q = RN(q1 + r1*y) is exactly RN(x/s) by Markstein's theorem (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990; the remainders are exact FMA
// results).  The preconditions hold whenever |x/s| >= 1/4 (no underflow);
// below that every quotient rounds to code 0 anyway.  Rows whose absmax is
// not finite take the oracle's literal IEEE-division path.
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

    __host__ __device__ static constexpr int stage_bytes(int T) { return (kStatePad + T * kTokBytes + 127) / 128 * 128; }
    __host__ __device__ static constexpr int region_bytes(int T) {
        int r = stage_bytes(T);
        r += T * kRowVecs * D * 4 + 64;  // row vectors, per-token decays and strengths (replay)
        if (kMixed) r += kWarps * D * 4 + D * 12 + 128;  // partials, s/-s/1/s, flag
        return (r + 127) / 128 * 128;
    }
};

__device__ __forceinline__ void report(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

constexpr float kRound = 12582912.0f;            // 1.5 * 2^23: x + kRound - kRound = rint(x)
constexpr float kCodeBias = 8388736.0f;          // 2^23 + 128

// Byte layout of a mixed tile (rows interleaved by 32-bit word inside each
// region; see the header): FP16 value (r, c) is half ((r/2)*D + c)*2 + r%2,
// INT8 value (r, c) is byte ((q/4)*D + c)*4 + q%4 with q = r - KH.  Thread c
// of a group therefore moves one column of 2 FP16 rows or 4 INT8 rows with a
// single 32-bit shared-memory access.

// Exact INT8 code for one value (IEEE division), the oracle's definition.
__device__ __forceinline__ uint32_t quant_exact(float x, float s) {
    float r = rintf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<uint32_t>(static_cast<int32_t>(r)) & 0xffu;
}

// INT8 codes of four values (one column of rows 4q..4q+3) of finite rows
// with scales s, negated scales ns = -s and reciprocals y = rcp_rn(s):
// q = RN(x/s) by two FMA corrections (see the top of this file), then
// round-half-even through the 1.5 * 2^23 addend; the low byte of each sum is
// the two's-complement code.  |q| <= 127.00002, so no clamp is needed.
__device__ __forceinline__ uint32_t quant_quad(float2 x01, float2 x23, float4 ns, float4 y) {
    const float2 y01 = make_float2(y.x, y.y), y23 = make_float2(y.z, y.w);
    const float2 n01 = make_float2(ns.x, ns.y), n23 = make_float2(ns.z, ns.w);
    float2 q01 = __fmul2_rn(x01, y01);
    float2 q23 = __fmul2_rn(x23, y23);
    q01 = __ffma2_rn(__ffma2_rn(q01, n01, x01), y01, q01);
    q23 = __ffma2_rn(__ffma2_rn(q23, n23, x23), y23, q23);
    q01 = __ffma2_rn(__ffma2_rn(q01, n01, x01), y01, q01);
    q23 = __ffma2_rn(__ffma2_rn(q23, n23, x23), y23, q23);
    const float2 m01 = __fadd2_rn(q01, make_float2(kRound, kRound));
    const float2 m23 = __fadd2_rn(q23, make_float2(kRound, kRound));
    const uint32_t lo2 = __byte_perm(__float_as_uint(m01.x), __float_as_uint(m01.y), 0x0040);
    const uint32_t hi2 = __byte_perm(__float_as_uint(m23.x), __float_as_uint(m23.y), 0x0040);
    return __byte_perm(lo2, hi2, 0x5410);
}

__device__ __forceinline__ uint32_t quant_quad_exact(float2 x01, float2 x23, float4 s) {
    return quant_exact(x01.x, s.x) | (quant_exact(x01.y, s.y) << 8) |
           (quant_exact(x23.x, s.z) << 16) | (quant_exact(x23.y, s.w) << 24);
}

// Fused arithmetic (RS_QUANT_FUSED): the code is the integer nearest to the
// exact product x * y, y = RN(1/s), rounded once -- the fused multiply-add
// x * y + 1.5 * 2^23 leaves it in the low mantissa bits (|x y| < 127.5, so
// the sum stays in [2^23, 2^24) where the spacing is 1).  The low byte of the
// sum is the two's-complement code.
__device__ __forceinline__ uint32_t quant_quad_rcp(float2 x01, float2 x23, float4 y) {
    const float2 m01 = __ffma2_rn(x01, make_float2(y.x, y.y), make_float2(kRound, kRound));
    const float2 m23 = __ffma2_rn(x23, make_float2(y.z, y.w), make_float2(kRound, kRound));
    const uint32_t lo2 = __byte_perm(__float_as_uint(m01.x), __float_as_uint(m01.y), 0x0040);
    const uint32_t hi2 = __byte_perm(__float_as_uint(m23.x), __float_as_uint(m23.y), 0x0040);
    return __byte_perm(lo2, hi2, 0x5410);
}

// One fused-arithmetic code of a row whose reciprocal is y, or -- for a row
// whose absmax is inf or NaN, marked by y = 0 -- the IEEE quotient by s.
__device__ __forceinline__ uint32_t quant_rcp_or_exact(float x, float s, float y) {
    return y != 0.0f ? (__float_as_uint(__fmaf_rn(x, y, kRound)) & 0xffu) : quant_exact(x, s);
}

template <bool FUSED>
__device__ __forceinline__ uint32_t quant_quad_cold(float2 x01, float2 x23, float4 s, float4 y) {
    if constexpr (FUSED)
        return quant_rcp_or_exact(x01.x, s.x, y.x) | (quant_rcp_or_exact(x01.y, s.y, y.y) << 8) |
               (quant_rcp_or_exact(x23.x, s.z, y.z) << 16) | (quant_rcp_or_exact(x23.y, s.w, y.w) << 24);
    else
        return quant_quad_exact(x01, x23, s);
}

// Dequantise column tid of a mixed tile (shared or global memory) into row
// pairs xs[j] = rows (2j, 2j+1).  int8 -> float is exact without a
// conversion instruction: the code byte, offset by 128, becomes the low
// mantissa byte of 2^23 and the bias is subtracted.  `scales` (16-byte
// aligned, D - KH floats) replaces the tile's own row scales when given.
template <int D, int KH>
__device__ __forceinline__ void mixed_dequant(const uint8_t *tile, int tid, float2 (&xs)[D / 2],
                                              const float *scales = nullptr) {
    const __half2 *hi = reinterpret_cast<const __half2 *>(tile);
    const uint32_t *lo = reinterpret_cast<const uint32_t *>(tile + 2 * KH * D);
    const float4 *sc4 = reinterpret_cast<const float4 *>(
        scales ? scales : reinterpret_cast<const float *>(tile + 2 * KH * D + (D - KH) * D));
#pragma unroll
    for (int j = 0; j < KH / 2; ++j) xs[j] = __half22float2(hi[j * D + tid]);
#pragma unroll
    for (int qd = 0; qd < (D - KH) / 4; ++qd) {
        const uint32_t w = lo[qd * D + tid] ^ 0x80808080u;
        const float4 s4 = sc4[qd];
        const float f0 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540));
        const float f1 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541));
        const float f2 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542));
        const float f3 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543));
        const float2 c01 = __fadd2_rn(make_float2(f0, f1), make_float2(-kCodeBias, -kCodeBias));
        const float2 c23 = __fadd2_rn(make_float2(f2, f3), make_float2(-kCodeBias, -kCodeBias));
        xs[KH / 2 + 2 * qd] = __fmul2_rn(c01, make_float2(s4.x, s4.y));
        xs[KH / 2 + 2 * qd + 1] = __fmul2_rn(c23, make_float2(s4.z, s4.w));
    }
}

// Per-row absmax bookkeeping: after a warp max-reduction of rows 2j and
// 2j+1, lane (r & 31) keeps the maximum of row r in mine[r >> 5].
template <int D>
__device__ __forceinline__ void absmax_pair(float2 xv, int j, int lane, float (&mine)[D / 32]) {
    const float m0 = warp_max_abs_nan(xv.x);
    const float m1 = warp_max_abs_nan(xv.y);
    mine[(2 * j) >> 5] = lane == ((2 * j) & 31) ? m0 : mine[(2 * j) >> 5];
    mine[(2 * j + 1) >> 5] = lane == ((2 * j + 1) & 31) ? m1 : mine[(2 * j + 1) >> 5];
}

// Requantise the FP32 column (row pairs xs, thread tid of a group of D
// threads, warp wig, lane lane) into a mixed tile assembled at `out` in
// shared memory (same byte layout as a pool tile), given the warp's per-row
// maxima in mine (see absmax_pair).  red ([D/32][D] floats), sc, nsc and rc
// ([D] floats each: row scale, its negation, its reciprocal) and flag (one
// int, zero on entry) are group-private scratch; bar_id/D name the group
// barrier.  `before_write` runs on every thread before the group barrier
// that precedes the first write into `out`.  Bit-exact with the oracle, in
// the IEEE (FUSED = false) or the fused arithmetic.
template <int D, int KH, bool FUSED, typename F>
__device__ __forceinline__ void mixed_requant_from_max(const float2 (&xs)[D / 2], const float (&mine)[D / 32],
                                                       uint8_t *out, float *red, float *sc, float *nsc,
                                                       float *rc, int *flag, int tid, int lane, int wig,
                                                       uint32_t bar_id, F before_write) {
    constexpr int W = D / 32;
    constexpr int NQ = (D - KH) / 4;
    static_assert(KH % 4 == 0 && (D - KH) % 4 == 0, "row blocks of four");
#pragma unroll
    for (int k = 0; k < D / 32; ++k)
        if (32 * k + lane >= KH) red[wig * D + 32 * k + lane] = mine[k];
    before_write();
    group_sync(bar_id, D);
    if (tid >= KH) {
        uint32_t ab = __float_as_uint(red[tid]);
#pragma unroll
        for (int w = 1; w < W; ++w) ab = max(ab, __float_as_uint(red[w * D + tid]));
        const float a = __uint_as_float(ab);  // >= 0, or NaN (largest bit pattern)
        const float s = __fdiv_rn(fmaxf(a, 1e-8f), 127.0f);
        sc[tid] = s;
        nsc[tid] = -s;
        // fused arithmetic: y = 0 marks a row whose absmax is inf or NaN
        rc[tid] = (FUSED && ab >= 0x7f800000u) ? 0.0f : __frcp_rn(s);
        if (ab >= 0x7f800000u) *flag = 1;  // absmax inf or NaN: exact path for the tile
        reinterpret_cast<float *>(out + 2 * KH * D + (D - KH) * D)[tid - KH] = s;
    }
    group_sync(bar_id, D);
    __half2 *hi = reinterpret_cast<__half2 *>(out);
#pragma unroll
    for (int j = 0; j < KH / 2; ++j) hi[j * D + tid] = __floats2half2_rn(xs[j].x, xs[j].y);
    uint32_t *lo = reinterpret_cast<uint32_t *>(out + 2 * KH * D);
    if (*flag == 0) {
        const float4 *rc4 = reinterpret_cast<const float4 *>(rc + KH);
        const float4 *ns4 = reinterpret_cast<const float4 *>(nsc + KH);
#pragma unroll
        for (int qd = 0; qd < NQ; ++qd) {
            if constexpr (FUSED)
                lo[qd * D + tid] = quant_quad_rcp(xs[KH / 2 + 2 * qd], xs[KH / 2 + 2 * qd + 1], rc4[qd]);
            else
                lo[qd * D + tid] = quant_quad(xs[KH / 2 + 2 * qd], xs[KH / 2 + 2 * qd + 1], ns4[qd], rc4[qd]);
        }
    } else {
        const float4 *sc4 = reinterpret_cast<const float4 *>(sc + KH);
        const float4 *rc4 = reinterpret_cast<const float4 *>(rc + KH);
#pragma unroll 1
        for (int qd = 0; qd < NQ; ++qd) {
            // dynamic quad index on this cold path: select the pair from the
            // register array without indexing it dynamically
            float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < NQ; ++k)
                if (k == qd) {
                    a01 = xs[KH / 2 + 2 * k];
                    a23 = xs[KH / 2 + 2 * k + 1];
                }
            lo[qd * D + tid] = quant_quad_cold<FUSED>(a01, a23, sc4[qd], rc4[qd]);
        }
    }
}

// Same, collecting the per-row maxima first (for callers that did not fuse
// the reductions into the update pass).
template <int D, int KH, bool FUSED, typename F>
__device__ __forceinline__ void mixed_requant_smem(const float2 (&xs)[D / 2], uint8_t *out, float *red,
                                                   float *sc, float *nsc, float *rc, int *flag,
                                                   int tid, int lane, int wig, uint32_t bar_id,
                                                   F before_write) {
    float mine[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) mine[k] = 0.0f;
#pragma unroll
    for (int j = KH / 2; j < D / 2; ++j) absmax_pair<D>(xs[j], j, lane, mine);
    mixed_requant_from_max<D, KH, FUSED>(xs, mine, out, red, sc, nsc, rc, flag, tid, lane, wig, bar_id,
                                         before_write);
}

// Dequantise rows 4q..4q+3 (q counted from row 0) of column tid of a mixed
// tile into two row pairs.
template <int D, int KH>
__device__ __forceinline__ void mixed_dequant_quad(const uint8_t *tile, int q, int tid, float2 &x01,
                                                   float2 &x23) {
    if (4 * q < KH) {
        const __half2 *hi = reinterpret_cast<const __half2 *>(tile);
        x01 = __half22float2(hi[(2 * q) * D + tid]);
        x23 = __half22float2(hi[(2 * q + 1) * D + tid]);
    } else {
        const int qd = q - KH / 4;
        const uint32_t *lo = reinterpret_cast<const uint32_t *>(tile + 2 * KH * D);
        const float4 *sc4 = reinterpret_cast<const float4 *>(tile + 2 * KH * D + (D - KH) * D);
        const uint32_t w = lo[qd * D + tid] ^ 0x80808080u;
        const float4 s4 = sc4[qd];
        const float f0 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540));
        const float f1 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541));
        const float f2 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542));
        const float f3 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543));
        x01 = __fmul2_rn(__fadd2_rn(make_float2(f0, f1), make_float2(-kCodeBias, -kCodeBias)),
                         make_float2(s4.x, s4.y));
        x23 = __fmul2_rn(__fadd2_rn(make_float2(f2, f3), make_float2(-kCodeBias, -kCodeBias)),
                         make_float2(s4.z, s4.w));
    }
}

template <int D, int KHI, bool KDA, int MAXT, typename TI, typename TO, typename PT, bool FUSED = false>
__global__ void __launch_bounds__(step_threads(MAXT), 1)
    step_kernel(const __grid_constant__ PT P) {
    using S = StepShape<D, KHI, KDA, TI>;
    constexpr bool MIXED = S::kMixed;
    constexpr int KH = S::kKhi;
    constexpr int DP = D / 2;  // row pairs per column

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
    float *rowv = reinterpret_cast<float *>(region + S::stage_bytes(T));
    // rowv layout per token t: [K | BK | Q | V | A?] each D floats
    float *tok_alpha = rowv + T * S::kRowVecs * D;                  // [8] GDN decays (replay)
    float *tok_beta = tok_alpha + 8;                                // [8] write strengths (replay)
    float *red = tok_beta + 8;                                      // [kWarps][D]   (mixed)
    float *scl = red + S::kWarps * D;                               // [D] row scales
    float *nscl = scl + D;                                          // [D] -scales
    float *rcp = nscl + D;                                          // [D] reciprocals
    int *flag = reinterpret_cast<int *>(rcp + D);                   // non-finite row seen

    if (threadIdx.x < G) mbar_init(&bars[threadIdx.x], 1);
    if constexpr (MIXED)
        for (int i = threadIdx.x; i < Hv * D; i += blockDim.x) pi_s[i] = P.pi[i];
    fence_mbar_init();
    pdl_launch_next();
    pdl_wait();  // the previous kernel's writes are visible from here on
    __syncthreads();

    uint64_t *bar = &bars[grp];
    const uint32_t bar_id = 1 + grp;
    const int items = P.B * Hv;
    const int gstride = gridDim.x * G;
    const TI *q_g = static_cast<const TI *>(P.q);
    const TI *k_g = static_cast<const TI *>(P.k);
    const TI *v_g = static_cast<const TI *>(P.v);
    uint8_t *pool = static_cast<uint8_t *>(P.pool);

    // (slot, accepted tokens) of an item; every thread of the group reads the
    // same words, one item ahead, so the load latency stays off the critical path.
    auto item_slot = [&](int it) -> int32_t { return it < items ? P.slot_idx[it / Hv] : -1; };
    auto item_n = [&](int it) -> int32_t {
        return it < items ? (P.replay ? P.n_accept[it / Hv] : 1) : 0;
    };

    // Producer step, run by thread 0 of the group: start the copies of item it.
    auto issue = [&](int it, int32_t slot, int32_t n) {
        if (it >= items || slot < 0 || (int64_t)slot >= P.n_slots || n < 1 || n > T) return;
        const int b = it / Hv, h = it - (it / Hv) * Hv;
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

    // Replay: thread t < n of the group holds token t's write strength (and
    // GDN decay) of the next item in registers, loaded one item ahead; they
    // reach shared memory at the start of that item.
    auto tok_scalars = [&](int it, int32_t n, float &bt, float &at) {
        bt = 0.0f;
        at = 0.0f;
        if (MAXT > 1 && tid < n && it < items) {
            const size_t bti = ((size_t)(it / Hv) * T + tid) * Hv + (it - (it / Hv) * Hv);
            bt = P.beta[bti];
            if (!KDA) at = P.alpha[bti];
        }
    };

    int item = blockIdx.x * G + grp;
    int32_t cur_slot = item_slot(item), cur_n = item_n(item);
    if (tid == 0) issue(item, cur_slot, cur_n);
    uint32_t phase = 0;
    float cur_bt, cur_at;
    tok_scalars(item, cur_n, cur_bt, cur_at);

    for (; item < items; item += gstride) {
        const int b = item / Hv, h = item - (item / Hv) * Hv;
        const int nxt = item + gstride;
        const int32_t nxt_slot = item_slot(nxt), nxt_n = item_n(nxt);
        const int32_t slot = cur_slot, n = cur_n;
        cur_slot = nxt_slot;
        cur_n = nxt_n;
        if (MAXT > 1 && tid < MAXT) {  // visible after the barrier below
            tok_beta[tid] = cur_bt;
            tok_alpha[tid] = cur_at;
        }
        if constexpr (MAXT > 1) {
            const int32_t nn = (nxt_n >= 0 && nxt_n <= T) ? nxt_n : 0;
            tok_scalars(nxt, nn, cur_bt, cur_at);
        }
        const bool slot_ok = slot >= 0 && (int64_t)slot < P.n_slots;
        const bool n_ok = n >= 0 && n <= T;
        if (!slot_ok || !n_ok || n == 0) {
            if (tid == 0) {
                if (!slot_ok) report(P.status, 1);
                else if (!n_ok) report(P.status, 2);
                issue(nxt, nxt_slot, nxt_n);
            }
            continue;
        }
        // Scalars of a single-token item, loaded before the wait so their
        // latency hides.  Replay instances took theirs one item ahead.
        float beta0 = 0.0f, alpha0 = 0.0f;
        if constexpr (MAXT == 1) {
            beta0 = P.beta[(size_t)b * Hv + h];
            if (!KDA) alpha0 = P.alpha[(size_t)b * Hv + h];
        }

        bool got = mbar_wait_bounded(bar, phase);
        if (!got) got = mbar_wait_bounded(bar, phase);  // copies still in flight get a second bound
        if (group_sync_or(bar_id, D, !got)) {
            if (tid == 0) report(P.status, 8);
            return;
        }
        phase ^= 1u;

        float2 x[DP];
        if constexpr (!MIXED) {
            // FP32 tile -> registers, then the stage can be refilled early.
            const float *st = reinterpret_cast<const float *>(stage);
#pragma unroll
            for (int j = 0; j < DP; ++j) x[j] = make_float2(st[(2 * j) * D + tid], st[(2 * j + 1) * D + tid]);
        }

        auto decay_of = [&](int t) -> float {
            return KDA ? 0.0f : (MAXT == 1 ? alpha0 : tok_alpha[t]);
        };
        // ---- token inputs -> per-row vectors (row u built by thread u) -----
        const int ntok = MAXT == 1 ? 1 : n;  // decode instances: one token, known at compile time
        {
            const int src = MIXED ? (int)pi_s[h * D + tid] : tid;
            for (int t = 0; t < ntok; ++t) {
                const uint8_t *tb = stage + S::kStatePad + t * S::kTokBytes;
                const TI *kt = reinterpret_cast<const TI *>(tb);
                const TI *qt = reinterpret_cast<const TI *>(tb + S::kVecBytes);
                const TI *vt = reinterpret_cast<const TI *>(tb + 2 * S::kVecBytes);
                float *rv = rowv + t * S::kRowVecs * D;
                const float kf = load_as_f32<TI>(kt + src);
                const float bt = MAXT == 1 ? beta0 : tok_beta[t];
                rv[tid] = kf;
                rv[D + tid] = __fmul_rn(bt, kf);
                rv[2 * D + tid] = load_as_f32<TI>(qt + src);
                rv[3 * D + tid] = load_as_f32<TI>(vt + tid);  // value coordinates: no row map
                const float at = KDA ? reinterpret_cast<const float *>(tb + 3 * S::kVecBytes)[src] : decay_of(t);
                if (KDA) rv[4 * D + tid] = at;
            }
        }
        group_sync(bar_id, D);  // row vectors visible (FP32: stage fully read)
        if constexpr (!MIXED) {
            if (tid == 0) {
                fence_proxy_async_smem();
                issue(nxt, nxt_slot, nxt_n);  // the stage now belongs to the next tile
            }
        }

        TO *og = static_cast<TO *>(P.o);
        float mine[D / 32];
#pragma unroll
        for (int k = 0; k < D / 32; ++k) mine[k] = 0.0f;
        if constexpr (MAXT == 1) {
            // ---- one token: decay and prediction (mixed: fused with the
            // dequantisation), then write and readout (mixed: fused with the
            // per-row maxima), so each FMA chain has independent work beside it
            float p = 0.0f;
            const float a_s = decay_of(0);
#pragma unroll
            for (int j = 0; j < DP; j += 2) {
                if constexpr (MIXED) mixed_dequant_quad<D, KH>(stage, j / 2, tid, x[j], x[j + 1]);
                const float4 kk = *reinterpret_cast<const float4 *>(rowv + 2 * j);
                float4 aa;
                if (KDA) aa = *reinterpret_cast<const float4 *>(rowv + 4 * D + 2 * j);
                else aa = make_float4(a_s, a_s, a_s, a_s);
                x[j] = __fmul2_rn(x[j], make_float2(aa.x, aa.y));
                x[j + 1] = __fmul2_rn(x[j + 1], make_float2(aa.z, aa.w));
                p = __fmaf_rn(x[j].x, kk.x, p);
                p = __fmaf_rn(x[j].y, kk.y, p);
                p = __fmaf_rn(x[j + 1].x, kk.z, p);
                p = __fmaf_rn(x[j + 1].y, kk.w, p);
            }
            if constexpr (MIXED) {
                group_sync(bar_id, D);  // stage fully read
                if (tid == 0) {
                    fence_proxy_async_smem();
                    issue(nxt, nxt_slot, nxt_n);  // the stage now belongs to the next tile
                }
            }
            const float e = __fsub_rn(rowv[3 * D + tid], p);
            float o = 0.0f;
#pragma unroll
            for (int j = 0; j < DP; j += 2) {
                const float4 bk = *reinterpret_cast<const float4 *>(rowv + D + 2 * j);
                const float4 qq = *reinterpret_cast<const float4 *>(rowv + 2 * D + 2 * j);
                x[j] = __ffma2_rn(make_float2(bk.x, bk.y), make_float2(e, e), x[j]);
                x[j + 1] = __ffma2_rn(make_float2(bk.z, bk.w), make_float2(e, e), x[j + 1]);
                o = __fmaf_rn(x[j].x, qq.x, o);
                o = __fmaf_rn(x[j].y, qq.y, o);
                o = __fmaf_rn(x[j + 1].x, qq.z, o);
                o = __fmaf_rn(x[j + 1].y, qq.w, o);
                if constexpr (MIXED) {
                    if (2 * j >= KH) {  // row maxima beside the readout chain
                        absmax_pair<D>(x[j], j, lane, mine);
                        absmax_pair<D>(x[j + 1], j + 1, lane, mine);
                    }
                }
            }
            if (og) store_from_f32<TO>(og + ((size_t)b * Hv + h) * D + tid, o);
        } else {
            // ---- replay: the state stays in registers across the tokens
            if constexpr (MIXED) {
                mixed_dequant<D, KH>(stage, tid, x);
                group_sync(bar_id, D);  // stage fully read
                if (tid == 0) {
                    fence_proxy_async_smem();
                    issue(nxt, nxt_slot, nxt_n);  // the stage now belongs to the next tile
                }
            }
            // Token t's readout chain and token t + 1's decay and prediction chain
            // read the same updated rows, so one pass over the registers carries
            // both (two independent chains per thread); each chain keeps its
            // ascending row order, so the result equals token-by-token steps.
            auto decay4 = [&](const float *rv, int t, int j) -> float4 {
                float4 aa;
                if (KDA) aa = *reinterpret_cast<const float4 *>(rv + 4 * D + 2 * j);
                else { const float a_s = decay_of(t); aa = make_float4(a_s, a_s, a_s, a_s); }
                return aa;
            };
            float p = 0.0f;
#pragma unroll
            for (int j = 0; j < DP; j += 2) {  // token 0: decay and prediction
                const float4 kk = *reinterpret_cast<const float4 *>(rowv + 2 * j);
                const float4 aa = decay4(rowv, 0, j);
                x[j] = __fmul2_rn(x[j], make_float2(aa.x, aa.y));
                x[j + 1] = __fmul2_rn(x[j + 1], make_float2(aa.z, aa.w));
                p = __fmaf_rn(x[j].x, kk.x, p);
                p = __fmaf_rn(x[j].y, kk.y, p);
                p = __fmaf_rn(x[j + 1].x, kk.z, p);
                p = __fmaf_rn(x[j + 1].y, kk.w, p);
            }
            for (int t = 0; t < ntok; ++t) {
                const float *rv = rowv + t * S::kRowVecs * D;
                const float e = __fsub_rn(rv[3 * D + tid], p);
                float o = 0.0f;
                if (t + 1 < ntok) {
                    const float *rn = rv + S::kRowVecs * D;  // token t + 1
                    float pn = 0.0f;
#pragma unroll
                    for (int j = 0; j < DP; j += 2) {
                        const float4 bk = *reinterpret_cast<const float4 *>(rv + D + 2 * j);
                        const float4 qq = *reinterpret_cast<const float4 *>(rv + 2 * D + 2 * j);
                        const float4 kk = *reinterpret_cast<const float4 *>(rn + 2 * j);
                        const float4 aa = decay4(rn, t + 1, j);
                        x[j] = __ffma2_rn(make_float2(bk.x, bk.y), make_float2(e, e), x[j]);
                        x[j + 1] = __ffma2_rn(make_float2(bk.z, bk.w), make_float2(e, e), x[j + 1]);
                        o = __fmaf_rn(x[j].x, qq.x, o);
                        o = __fmaf_rn(x[j].y, qq.y, o);
                        o = __fmaf_rn(x[j + 1].x, qq.z, o);
                        o = __fmaf_rn(x[j + 1].y, qq.w, o);
                        x[j] = __fmul2_rn(x[j], make_float2(aa.x, aa.y));
                        x[j + 1] = __fmul2_rn(x[j + 1], make_float2(aa.z, aa.w));
                        pn = __fmaf_rn(x[j].x, kk.x, pn);
                        pn = __fmaf_rn(x[j].y, kk.y, pn);
                        pn = __fmaf_rn(x[j + 1].x, kk.z, pn);
                        pn = __fmaf_rn(x[j + 1].y, kk.w, pn);
                    }
                    p = pn;
                } else {
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
                }
                if (og) store_from_f32<TO>(og + (((size_t)b * T + t) * Hv + h) * D + tid, o);
            }
            if constexpr (MIXED) {
#pragma unroll
                for (int j = KH / 2; j < DP; ++j) absmax_pair<D>(x[j], j, lane, mine);
            }
        }

        // ---- registers -> HBM ---------------------------------------------
        uint8_t *tile = pool + ((size_t)slot * Hv + h) * S::kStateBytes;
        if constexpr (!MIXED && MAXT == 1) {
            // Rows 4r..4r+3 of the four columns of a lane quad are transposed
            // among its lanes (two exchanges), so lane i stores row 4r + i of
            // the quad's columns as one 16-byte store: a warp writes four
            // whole 128-byte row segments per instruction.  (Replay, whose
            // threads hold more registers, keeps the column stores: the
            // exchanges cost it more than the wider stores save.)
            float *st = reinterpret_cast<float *>(tile);
            const bool b0 = tid & 1, b1 = tid & 2;
#pragma unroll
            for (int r = 0; r < DP / 2; ++r) {
                const float a0 = x[2 * r].x, a1 = x[2 * r].y, a2 = x[2 * r + 1].x, a3 = x[2 * r + 1].y;
                // exchange 1 (lanes i, i ^ 2): rows 2, 3 for rows 0, 1 of the partner
                const float r0 = __shfl_xor_sync(0xffffffffu, b1 ? a0 : a2, 2);
                const float r1 = __shfl_xor_sync(0xffffffffu, b1 ? a1 : a3, 2);
                const float l0 = b1 ? r0 : a0, l1 = b1 ? r1 : a1, l2 = b1 ? a2 : r0, l3 = b1 ? a3 : r1;
                // exchange 2 (lanes i, i ^ 1)
                const float u0 = __shfl_xor_sync(0xffffffffu, b0 ? l0 : l1, 1);
                const float u1 = __shfl_xor_sync(0xffffffffu, b0 ? l2 : l3, 1);
                const float4 w = b0 ? make_float4(u0, l1, u1, l3) : make_float4(l0, u0, l2, u1);
                *reinterpret_cast<float4 *>(st + (4 * r + (tid & 3)) * D + (tid & ~3)) = w;
            }
        } else if constexpr (!MIXED) {
            float *st = reinterpret_cast<float *>(tile);
#pragma unroll
            for (int j = 0; j < DP; ++j) {
                st[(2 * j) * D + tid] = x[j].x;
                st[(2 * j + 1) * D + tid] = x[j].y;
            }
        } else {
            // the requantised words go from registers straight to the tile in HBM
            // (thread tid writes column tid of each word row: 128 contiguous bytes a warp)
            mixed_requant_from_max<D, KH, FUSED>(x, mine, tile, red, scl, nscl, rcp, flag, tid, lane, wig,
                                                 bar_id, [&] {
                                                     if (tid == 0) *flag = 0;
                                                 });
        }
        group_sync(bar_id, D);  // row vectors / partials free for the next item
    }
}

}  // namespace rs
