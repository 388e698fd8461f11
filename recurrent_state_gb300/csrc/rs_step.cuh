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
//     is held as row pairs, and the dequantise / requantise arithmetic of the
//     mixed layout runs as paired FP32 instructions (mul/add/fma .f32x2), two
//     rows per instruction, each lane rounded on its own;
//   * a replay keeps the state on chip across tokens ("Serving recurrent
//     attention", speculative decoding without state snapshots).
// The tile and the token inputs arrive through a 1-D bulk TMA copy
// (cp.async.bulk + mbarrier) into the group's shared-memory stage; as soon as
// the stage has been read into registers the group issues the copy of its
// next tile, so HBM reads of tile i+1 overlap the arithmetic of tile i.
// FP32 tiles go straight from registers to HBM with coalesced stores (a warp
// writes 32 consecutive columns of a row); mixed tiles are assembled in a
// shared-memory staging buffer and written with one bulk TMA store.
//
// Mixed layout (DAMP §5.2, Appendix A.4): FP16 rows and INT8 rows with one
// FP32 scale per row are dequantised into the registers, updated in FP32, and
// requantised in the same pass; the per-row absmax is a warp max-reduction
// (redux.sync) plus a combine over the group's warps in shared memory.  The
// INT8 code is round_half_even(x / s) with x / s the IEEE quotient: the
// kernel computes q0 = x * rcp_rn(s); since |q0 - fl(x/s)| <= 3 * 2^-24 *
// |x/s| < 2^-15 for |x/s| <= 127.0001, every q0 farther than 2^-15 from a
// half-integer rounds like fl(x/s); the rest (about 6e-5 of the values) take
// the exact IEEE division.
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
        r += T * kRowVecs * D * 4;
        if (kMixed) r += kWarps * D * 4 + D * 8 + kStatePad;  // absmax partials, (s, 1/s), out tile
        return (r + 127) / 128 * 128;
    }
};

__device__ __forceinline__ void report(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

constexpr float kRound = 12582912.0f;            // 1.5 * 2^23: x + kRound - kRound = rint(x)
constexpr float kNearHalf = 0.499969482421875f;  // 0.5 - 2^-15

// Exact INT8 code for one value on the slow path (IEEE division).
__device__ __forceinline__ uint32_t quant_exact(float x, float s) {
    float r = rintf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<uint32_t>(static_cast<int32_t>(r));
}

// INT8 codes of two values x (rows r, r+1) with scales s and reciprocals
// y = rcp_rn(s) (NaN marks a row whose absmax is not finite).  The low byte
// of each result is the two's-complement code.
__device__ __forceinline__ void quant_pair(float2 x, float2 s, float2 y, uint32_t &c0,
                                           uint32_t &c1) {
    const float2 q0 = __fmul2_rn(x, y);
    const float2 m = __fadd2_rn(q0, make_float2(kRound, kRound));
    const float2 rr = __fadd2_rn(m, make_float2(-kRound, -kRound));
    const float2 t = __ffma2_rn(rr, make_float2(-1.0f, -1.0f), q0);  // q0 - rint(q0), exact
    float tm;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(tm) : "f"(fabsf(t.x)), "f"(fabsf(t.y)));
    if (tm < kNearHalf) {
        c0 = __float_as_uint(m.x);
        c1 = __float_as_uint(m.y);
    } else {
        c0 = quant_exact(x.x, s.x);
        c1 = quant_exact(x.y, s.y);
    }
}

// Dequantise column tid of a mixed tile (shared or global memory) into row
// pairs xs[j] = rows (2j, 2j+1).  int8 -> float uses the exact magic-number
// form (c + 0x4B400000 as float) - 1.5 * 2^23 instead of a conversion.
template <int D, int KH>
__device__ __forceinline__ void mixed_dequant(const uint8_t *tile, int tid, float2 (&xs)[D / 2]) {
    const __half *hi = reinterpret_cast<const __half *>(tile);
    const int8_t *lo = reinterpret_cast<const int8_t *>(tile + 2 * KH * D);
    const float4 *sc4 = reinterpret_cast<const float4 *>(tile + 2 * KH * D + (D - KH) * D);
#pragma unroll
    for (int j = 0; j < KH / 2; ++j)
        xs[j] = make_float2(__half2float(hi[(2 * j) * D + tid]), __half2float(hi[(2 * j + 1) * D + tid]));
#pragma unroll
    for (int j = KH / 2; j < D / 2; j += 2) {  // four INT8 rows per step: one float4 of scales
        const int r = 2 * j - KH;
        const float4 s4 = sc4[r / 4];
        const int c0 = lo[(r + 0) * D + tid], c1 = lo[(r + 1) * D + tid];
        const int c2 = lo[(r + 2) * D + tid], c3 = lo[(r + 3) * D + tid];
        const float2 f01 = __fadd2_rn(make_float2(__int_as_float(c0 + 0x4B400000), __int_as_float(c1 + 0x4B400000)),
                                      make_float2(-kRound, -kRound));
        const float2 f23 = __fadd2_rn(make_float2(__int_as_float(c2 + 0x4B400000), __int_as_float(c3 + 0x4B400000)),
                                      make_float2(-kRound, -kRound));
        xs[j] = __fmul2_rn(f01, make_float2(s4.x, s4.y));
        xs[j + 1] = __fmul2_rn(f23, make_float2(s4.z, s4.w));
    }
}

// Requantise the FP32 column (row pairs xs, thread tid of a group of D
// threads, warp wig, lane lane) into a mixed tile assembled at `out` in
// shared memory (same byte layout as a pool tile).  red ([D/32][D] floats)
// and sy ([D] float2) are group-private scratch; bar_id/D name the group
// barrier.  `before_write` runs on every thread after the absmax phase and
// before the group barrier that precedes the first write into `out`.
// Matches the oracle's quantiser bit for bit.
template <int D, int KH, typename F>
__device__ __forceinline__ void mixed_requant_smem(const float2 (&xs)[D / 2], uint8_t *out, float *red,
                                                   float2 *sy, int tid, int lane, int wig,
                                                   uint32_t bar_id, F before_write) {
    constexpr int W = D / 32;
    static_assert(KH % 4 == 0 && (D - KH) % 4 == 0, "row blocks of four");
    // per-row absmax: one warp max-reduction per row; lane (r & 31) keeps row r
    float mine[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) mine[k] = 0.0f;
#pragma unroll
    for (int j = KH / 2; j < D / 2; ++j) {
        const float m0 = warp_max_abs_nan(xs[j].x);
        const float m1 = warp_max_abs_nan(xs[j].y);
        if (lane == ((2 * j) & 31)) mine[(2 * j) >> 5] = m0;
        if (lane == ((2 * j + 1) & 31)) mine[(2 * j + 1) >> 5] = m1;
    }
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
        const bool finite = ab < 0x7f800000u;
        sy[tid] = make_float2(s, finite ? __frcp_rn(s) : __int_as_float(0x7fc00000));
        reinterpret_cast<float *>(out + 2 * KH * D + (D - KH) * D)[tid - KH] = s;
    }
    group_sync(bar_id, D);
    __half *hi = reinterpret_cast<__half *>(out);
#pragma unroll
    for (int j = 0; j < KH / 2; ++j) {
        hi[(2 * j) * D + tid] = __float2half_rn(xs[j].x);
        hi[(2 * j + 1) * D + tid] = __float2half_rn(xs[j].y);
    }
    uint8_t *lo = out + 2 * KH * D;
    const float4 *sy4 = reinterpret_cast<const float4 *>(sy);
#pragma unroll
    for (int j = KH / 2; j < D / 2; ++j) {
        const float4 v = sy4[j];  // s_r, y_r, s_{r+1}, y_{r+1} for r = 2j
        uint32_t c0, c1;
        quant_pair(xs[j], make_float2(v.x, v.z), make_float2(v.y, v.w), c0, c1);
        lo[(2 * j - KH) * D + tid] = static_cast<uint8_t>(c0 & 0xffu);
        lo[(2 * j + 1 - KH) * D + tid] = static_cast<uint8_t>(c1 & 0xffu);
    }
}

template <int D, int KHI, bool KDA, int MAXT, typename TI, typename TO, typename PT>
__global__ void __launch_bounds__(kStepThreads, 1)
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
    float *red = rowv + T * S::kRowVecs * D;                        // [kWarps][D]   (mixed)
    float2 *sy = reinterpret_cast<float2 *>(red + S::kWarps * D);   // [D]           (mixed)
    uint8_t *outt = reinterpret_cast<uint8_t *>(sy + D);            // out tile      (mixed)

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

    int item = blockIdx.x * G + grp;
    int32_t cur_slot = item_slot(item), cur_n = item_n(item);
    if (tid == 0) issue(item, cur_slot, cur_n);
    uint32_t phase = 0;

    for (; item < items; item += gstride) {
        const int b = item / Hv, h = item - (item / Hv) * Hv;
        const int nxt = item + gstride;
        const int32_t nxt_slot = item_slot(nxt), nxt_n = item_n(nxt);
        const int32_t slot = cur_slot, n = cur_n;
        cur_slot = nxt_slot;
        cur_n = nxt_n;
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
            if (tid == 0) {
                report(P.status, 8);
                if constexpr (MIXED) bulk_store_wait_all();
            }
            return;
        }
        phase ^= 1u;

        // ---- state tile -> registers (row pairs) --------------------------
        float2 x[DP];
        if constexpr (!MIXED) {
            const float *st = reinterpret_cast<const float *>(stage);
#pragma unroll
            for (int j = 0; j < DP; ++j) x[j] = make_float2(st[(2 * j) * D + tid], st[(2 * j + 1) * D + tid]);
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
            issue(nxt, nxt_slot, nxt_n);  // the stage now belongs to the next tile
        }

        // ---- the recurrence, token by token, state in registers -----------
        const int ntok = MAXT == 1 ? 1 : n;  // decode instances: one token, known at compile time
        for (int t = 0; t < ntok; ++t) {
            const float *rv = rowv + t * S::kRowVecs * D;
            float a_s = 0.0f;
#pragma unroll
            for (int tt = 0; tt < MAXT; ++tt)
                if (tt == t) a_s = alpha_r[tt];
            // S <- diag(alpha) S ;  p = S^T k  (ascending rows)
            float p = 0.0f;
#pragma unroll
            for (int j = 0; j < DP; j += 2) {
                const float4 kk = *reinterpret_cast<const float4 *>(rv + 2 * j);
                float4 aa;
                if (KDA) aa = *reinterpret_cast<const float4 *>(rv + 4 * D + 2 * j);
                else aa = make_float4(a_s, a_s, a_s, a_s);
                x[j].x = __fmul_rn(x[j].x, aa.x);
                p = __fmaf_rn(x[j].x, kk.x, p);
                x[j].y = __fmul_rn(x[j].y, aa.y);
                p = __fmaf_rn(x[j].y, kk.y, p);
                x[j + 1].x = __fmul_rn(x[j + 1].x, aa.z);
                p = __fmaf_rn(x[j + 1].x, kk.z, p);
                x[j + 1].y = __fmul_rn(x[j + 1].y, aa.w);
                p = __fmaf_rn(x[j + 1].y, kk.w, p);
            }
            const float e = __fsub_rn(rv[3 * D + tid], p);
            // S <- S + beta k e^T ;  o = S^T q  (ascending rows)
            float o = 0.0f;
#pragma unroll
            for (int j = 0; j < DP; j += 2) {
                const float4 bk = *reinterpret_cast<const float4 *>(rv + D + 2 * j);
                const float4 qq = *reinterpret_cast<const float4 *>(rv + 2 * D + 2 * j);
                x[j].x = __fmaf_rn(bk.x, e, x[j].x);
                o = __fmaf_rn(x[j].x, qq.x, o);
                x[j].y = __fmaf_rn(bk.y, e, x[j].y);
                o = __fmaf_rn(x[j].y, qq.y, o);
                x[j + 1].x = __fmaf_rn(bk.z, e, x[j + 1].x);
                o = __fmaf_rn(x[j + 1].x, qq.z, o);
                x[j + 1].y = __fmaf_rn(bk.w, e, x[j + 1].y);
                o = __fmaf_rn(x[j + 1].y, qq.w, o);
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
            for (int j = 0; j < DP; ++j) {
                st[(2 * j) * D + tid] = x[j].x;
                st[(2 * j + 1) * D + tid] = x[j].y;
            }
        } else {
            mixed_requant_smem<D, KH>(x, outt, red, sy, tid, lane, wig, bar_id, [&] {
                if (tid == 0) bulk_store_wait_read();  // the previous tile's store has read `outt`
            });
            fence_proxy_async_smem();  // this thread's writes to `outt` before the bulk store
            group_sync(bar_id, D);
            if (tid == 0) {
                bulk_s2g(tile, outt, S::kStateBytes);
                bulk_store_commit();
            }
        }
        group_sync(bar_id, D);  // row vectors / partials free for the next item
    }
    if constexpr (MIXED)
        if (tid == 0) bulk_store_wait_all();
}

}  // namespace rs
