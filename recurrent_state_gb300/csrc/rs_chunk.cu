// rs_chunk.cu -- prefill chunks in the chunk-parallel form on the tensor
// cores (sm_103a, FP32 state layout).
//
// DAMP Appendix A.4 "Prefill path" (prefill runs FP32 arithmetic within a
// chunk) and "Serving recurrent attention", "Kernels follow the serving
// phase" (prefill exposes parallel work across a chunk's tokens).  The
// recurrence of DAMP §3.1 Eq. 1-2 over C tokens, started from state S0
// (rows u = key channels, columns v = value dimensions), is evaluated as
//     Gamma_t  = prod_{s<=t} diag(alpha_s)             (cumulative decay)
//     A[t][i]  = sum_c k_t[c] k_i[c] prod_{s=i+1..t} alpha_s[c]     (i < t)
//     Bm[t][i] = sum_c q_t[c] k_i[c] prod_{s=i+1..t} alpha_s[c]     (i <= t)
//     R        = diag(beta) (V - Khat S0),   Khat[t] = Gamma_t k_t
//     W        = (I + diag(beta) A)^{-1} R   (the rows the tokens write)
//     O        = Qhat S0 + Bm W,             Qhat[t] = Gamma_t q_t
//     S_C      = Gamma_C S0 + Ktil^T W,      Ktil[i] = k_i prod_{s=i+1..C} alpha_s
// (the same map as C decode steps; tests/test_chunk_form.py checks the
// algebra against the oracle's recurrence).  Every decay product is a
// product of alphas in (0, 1], so nothing overflows whatever the decays.
//
// One CTA of 256 threads per SM takes (sequence, head) tiles in turn; the
// two threads v and v + 128 share value column v, which is tensor-memory
// lane v of every M = 128 product below (each takes half of the column's
// key channels or tokens).  The state lives in tensor memory as S^T (lane v, columns
// u) across the chunks of a tile.  Per chunk of C = 16 tokens:
//   MMA 1   [P^T | Oq^T] = S0^T [Khat ; Qhat]^T      (K = 128, N = 2C)
//   MMA 2   W^T = R^T T^T, T = (I + diag(beta) A)^{-1}  (K = C, N = C)
//   MMA 3   O^T = Oq^T + W^T Bm^T                      (K = C, N = C)
//   MMA 4   S_C^T = Gamma_C S0^T + W^T Ktil             (K = C, N = 128)
// all of kind::tf32 with each fp32 operand split into a tf32 high part and
// an exact remainder (three products: hi*hi + hi*lo + lo*hi, about 2^-21
// relative), fp32 accumulation in tensor memory.  The C x C matrices A, Bm
// and the unit lower triangular inverse T run on the CUDA cores while MMA 1
// runs: A[t][i] = Khat_t . Kchk_i and Bm[t][i] = Qhat_t . Kchk_i with
// Kchk_i = k_i / Gamma_i (the decay products factor through the cumulative
// decay), unless some cumulative decay of the chunk falls below 1e-30, where
// each pair takes the running product of its decays instead.  The result equals the token-by-token recurrence up to rounding (not
// bit for bit: the order of the sums differs).
#include "rs_internal.h"
#include "rs_device.cuh"
#include "rs_tc.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

__device__ __forceinline__ void report_bits(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

constexpr int D = 128;        // dk = dv
constexpr int C = 16;         // tokens per chunk
constexpr int kThreads = 256;  // two threads per value column
constexpr uint32_t kTmemCols = 256;

// shared memory (bytes): tf32 operands in the K-major core-matrix layout of
// rs_tc.cuh, hi and lo parts; staged token inputs; small matrices
constexpr int kSA = D * D * 4;      // S0^T (M = v, K = u)
constexpr int kB1 = 2 * C * D * 4;  // [Khat ; Qhat] (N = 2C, K = u)
constexpr int kCC = C * C * 4;      // T or Bm (N = t, K = i)
constexpr int kKT = D * C * 4;      // Ktil^T (N = c, K = i)
constexpr int kA2 = D * C * 4;      // R^T, then W^T (M = v, K = t)
constexpr int DP = D + 4;           // padded row of the staged token vectors (bank spread)
constexpr int kTok = C * DP * 4;    // k, q or alpha of the chunk, [t][c] fp32
constexpr int oSAh = 0, oSAl = oSAh + kSA, oB1h = oSAl + kSA, oB1l = oB1h + kB1;
constexpr int oTh = oB1l + kB1, oTl = oTh + kCC, oBh = oTl + kCC, oBl = oBh + kCC;
constexpr int oKTh = oBl + kCC, oKTl = oKTh + kKT, oA2h = oKTl + kKT, oA2l = oA2h + kA2;
constexpr int oK = oA2l + kA2, oQ = oK + kTok, oAl = oQ + kTok;
constexpr int oBeta = oAl + kTok, oGc = oBeta + C * 4, oMA = oGc + D * 4, oMB = oMA + kCC;
constexpr int oBar = oMB + kCC, oTslot = oBar + 5 * 8, oAlpS = oTslot + 16;
constexpr int kSmemEnd = oAlpS + C * 4;
constexpr int kSmem = kSmemEnd;
static_assert(kSmem <= 232448, "fits the shared memory of one SM");
static_assert(oBar % 8 == 0 && oSAl % 1024 == 0 && oB1h % 16 == 0, "alignment");

// tensor-memory columns: S^T [0, 128), P^T [128, 128 + C), Oq^T [.., + C), W^T [.., + C)
constexpr uint32_t cS = 0, cP = D, cOq = D + C, cW = D + 2 * C;

// store x as a tf32 pair (hi, exact remainder) at byte offset off of the two buffers
__device__ __forceinline__ void put_split(uint8_t *hi, uint8_t *lo, uint32_t off, float x) {
    const float h = tc::tf32_hi(x);
    *reinterpret_cast<float *>(hi + off) = h;
    *reinterpret_cast<float *>(lo + off) = x - h;
}
// four consecutive K values of one row (16 bytes, off 16-aligned)
__device__ __forceinline__ void put_split4(uint8_t *hi, uint8_t *lo, uint32_t off, float a, float b, float c,
                                           float d) {
    const float4 h = make_float4(tc::tf32_hi(a), tc::tf32_hi(b), tc::tf32_hi(c), tc::tf32_hi(d));
    *reinterpret_cast<float4 *>(hi + off) = h;
    *reinterpret_cast<float4 *>(lo + off) = make_float4(a - h.x, b - h.y, c - h.z, d - h.w);
}

template <bool KDA, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads, 1) chunk_prefill_kernel(const __grid_constant__ PrefillParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, w = tid >> 5;
    const int v = tid & (D - 1);  // value column (and key channel c in the per-channel work)
    const int hf = tid >> 7;      // which half of the column's channels / tokens
    float *kS = reinterpret_cast<float *>(smem + oK);   // [t][DP]: k, then Khat (fast form)
    float *qS = reinterpret_cast<float *>(smem + oQ);   // [t][DP]: q, then Qhat (fast form)
    float *aS = reinterpret_cast<float *>(smem + oAl);  // [t][DP]: alpha, then Kchk (fast form)
    float *betaS = reinterpret_cast<float *>(smem + oBeta);
    float *gC = reinterpret_cast<float *>(smem + oGc);
    float *mA = reinterpret_cast<float *>(smem + oMA);
    float *mB = reinterpret_cast<float *>(smem + oMB);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + oBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + oTslot);

    if (tid == 0)
        for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);  // MMA 1, MMA 2, MMA 3+4, state, inputs
    fence_mbar_init();
    if (w == 0) {
        tc::tmem_alloc(tslot, kTmemCols);
        tc::tmem_relinquish();
    }
    pdl_launch_next();
    pdl_wait();  // the previous kernel's writes are visible from here on
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *tslot + ((uint32_t)(32 * (w & 3)) << 16);  // this warp's 32 lanes
    // operand descriptors at k-step 0; step s is 256 s bytes on, i.e. + 16 s in the address field
    const uint64_t dSAh = tc::smem_desc(smem + oSAh, 128, D * 32), dSAl = tc::smem_desc(smem + oSAl, 128, D * 32);
    const uint64_t dB1h = tc::smem_desc(smem + oB1h, 128, D * 32), dB1l = tc::smem_desc(smem + oB1l, 128, D * 32);
    const uint64_t dA2h = tc::smem_desc(smem + oA2h, 128, C * 32), dA2l = tc::smem_desc(smem + oA2l, 128, C * 32);
    const uint64_t dTh = tc::smem_desc(smem + oTh, 128, C * 32), dTl = tc::smem_desc(smem + oTl, 128, C * 32);
    const uint64_t dBh = tc::smem_desc(smem + oBh, 128, C * 32), dBl = tc::smem_desc(smem + oBl, 128, C * 32);
    const uint64_t dKTh = tc::smem_desc(smem + oKTh, 128, C * 32), dKTl = tc::smem_desc(smem + oKTl, 128, C * 32);

    const int Hv = P.Hv, Hk = P.Hk, L = P.L;
    const int items = P.B * Hv;
    const TI *q_g = static_cast<const TI *>(P.q);
    const TI *k_g = static_cast<const TI *>(P.k);
    const TI *v_g = static_cast<const TI *>(P.v);
    TO *o_g = static_cast<TO *>(P.o);
    uint32_t ph = 0;  // parity of the three barriers: each completes once per chunk
    bool failed = false;

    auto wait = [&](int k) -> bool {
        const bool ok = mbar_wait_bounded(&bars[k], ph) || mbar_wait_bounded(&bars[k], ph);
        return __syncthreads_and(ok);
    };
    // the first tile at or after `from` that this CTA processes (slot in range, 1 <= n <= L)
    auto next_work = [&](int from) -> int {
        for (int it = from; it < items; it += gridDim.x) {
            const int bb = it / Hv;
            const int32_t sl = P.slot_idx[bb];
            const int32_t nn = P.n_tokens ? P.n_tokens[bb] : L;
            if (sl >= 0 && (int64_t)sl < P.n_slots && nn >= 1 && nn <= L) return it;
        }
        return items;
    };
    // bulk copy of a tile's state ([u][v] row-major, 64 KB) into the lo operand buffer, staged
    auto prefetch_state = [&](int it) {
        if (tid != 0 || it >= items) return;
        const int bb = it / Hv, hh = it - bb * Hv;
        const float *src = static_cast<const float *>(P.pool) + ((size_t)P.slot_idx[bb] * Hv + hh) * D * D;
        mbar_arrive_expect_tx(&bars[3], (uint32_t)(D * D * 4));
        for (int part = 0; part < 4; ++part)
            bulk_g2s(smem + oSAl + part * (D * D), src + part * (D * D / 4), D * D, &bars[3]);
    };
    // a group's token vectors by bulk copies into the [Khat ; Qhat] operand buffers (free from
    // the end of MMA 1 to the next group's decays), raw: k, q, v [C][D] TI, then (KDA) alpha
    // [C][D] fp32; the per-token scalars (beta, GDN alpha) into registers of threads t < C
    constexpr uint32_t kVecTI = D * (uint32_t)sizeof(TI);
    const uint8_t *rawK = smem + oB1h, *rawQ = rawK + C * kVecTI, *rawV = rawQ + C * kVecTI;
    const float *rawA = reinterpret_cast<const float *>(rawV + C * kVecTI);
    static_assert(3 * C * D * sizeof(TI) + (KDA ? C * D * 4 : 0) <= 2 * kB1, "raw inputs fit the operand buffers");
    float fb = 0.0f, fga = 1.0f;  // beta and the GDN decay of token tid of the fetched group
    int fnt = 0;                  // tokens in the fetched group
    auto fetch = [&](int it, int tb) {
        const int bb = it / Hv, hh = it - bb * Hv, gg = hh / (Hv / Hk);
        const int nn = P.n_tokens ? P.n_tokens[bb] : L;
        const int ntt = min(C, nn - tb);
        fnt = ntt;
        // one copy per thread, spread over the warps (lanes 0..7 of each: the copies of one
        // warp issue one after another): thread (warp x, lane y < 8) copies vector x / 2 of
        // token 8 (x % 2) + y (0: k, 1: q, 2: v, 3: alpha)
        if (tid == 0) mbar_arrive_expect_tx(&bars[4], (uint32_t)ntt * (3 * kVecTI + (KDA ? D * 4 : 0)));
        __syncthreads();  // the expected bytes are set before any copy can complete
        {
            const int y = tid & 31, vec = w >> 1, t = 8 * (w & 1) + y;
            if (y < 8 && t < ntt && (KDA || vec < 3)) {
                const size_t bt = (size_t)bb * L + tb + t;
                if (vec == 0) bulk_g2s(smem + oB1h + t * kVecTI, k_g + (bt * Hk + gg) * D, kVecTI, &bars[4]);
                else if (vec == 1)
                    bulk_g2s(smem + oB1h + (C + t) * kVecTI, q_g + (bt * Hk + gg) * D, kVecTI, &bars[4]);
                else if (vec == 2)
                    bulk_g2s(smem + oB1h + (2 * C + t) * kVecTI, v_g + (bt * Hv + hh) * D, kVecTI, &bars[4]);
                else
                    bulk_g2s(smem + oB1h + 3 * C * kVecTI + t * D * 4, P.alpha + (bt * Hv + hh) * D, D * 4,
                             &bars[4]);
            }
        }
        fb = 0.0f, fga = 1.0f;
        if (tid < ntt) {
            const size_t bt = (size_t)bb * L + tb + tid;
            fb = P.beta[bt * Hv + hh];
            if (!KDA) fga = P.alpha[bt * Hv + hh];
        }
    };
    uint32_t iph = 0;  // parity of the input-copy barrier
    float *alpS = reinterpret_cast<float *>(smem + oAlpS);
    uint32_t sph = 0;  // parity of the state-copy barrier
    int staged = next_work(blockIdx.x);
    prefetch_state(staged);
    if (staged < items) fetch(staged, 0);

    for (int item = blockIdx.x; item < items && !failed; item += gridDim.x) {
        const int b = item / Hv, h = item - b * Hv;
        const int32_t slot = P.slot_idx[b];
        const int32_t n = P.n_tokens ? P.n_tokens[b] : L;
        // every thread sees the same item: the skips are uniform
        if (slot < 0 || (int64_t)slot >= P.n_slots) {
            if (tid == 0) report_bits(P.status, 1);
            continue;
        }
        if (n < 0 || n > L) {
            if (tid == 0) report_bits(P.status, 2);
            continue;
        }
        if (n == 0) continue;
        float *Sg = static_cast<float *>(P.pool) + ((size_t)slot * Hv + h) * D * D;
        // the following tile's slot and token count, read now (used by the last group)
        const int nxi = item + gridDim.x;
        const int32_t nx_slot = nxi < items ? P.slot_idx[nxi / Hv] : -1;
        const int32_t nx_n = nxi < items ? (P.n_tokens ? P.n_tokens[nxi / Hv] : L) : 0;

        for (int t0 = 0; t0 < n && !failed; t0 += C) {
            const int nt = min(C, n - t0);
            // ---- the chunk's inputs, copied in during the previous group (or at start): raw
            // vectors to padded fp32 rows (pads: k = q = 0, alpha = 1, v = 0, beta = 0)
            float vt[C / 2];
            {
                if (tid < C) {
                    betaS[tid] = fb;
                    alpS[tid] = fga;
                }
                const bool ok = mbar_wait_bounded(&bars[4], iph) || mbar_wait_bounded(&bars[4], iph);
                if (!__syncthreads_and(ok)) {
                    failed = true;
                    break;
                }
                iph ^= 1u;
#pragma unroll
                for (int j = 0; j < C / 2; ++j) {
                    const int t = (C / 2) * hf + j;
                    const bool real = t < nt;
                    kS[t * DP + v] = real ? load_as_f32<TI>(reinterpret_cast<const TI *>(rawK + t * kVecTI) + v) : 0.0f;
                    qS[t * DP + v] = real ? load_as_f32<TI>(reinterpret_cast<const TI *>(rawQ + t * kVecTI) + v) : 0.0f;
                    vt[j] = real ? load_as_f32<TI>(reinterpret_cast<const TI *>(rawV + t * kVecTI) + v) : 0.0f;
                    if constexpr (KDA) aS[t * DP + v] = real ? rawA[t * D + v] : 1.0f;
                    else aS[t * DP + v] = alpS[t];  // 1 for pads
                }
            }
            __syncthreads();
            // ---- channel c = v: cumulative decays Gamma_t[c]; the factored form if none is tiny
            const int c = v;
            float gam[C];
            {
                float pg = 1.0f;
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    pg = __fmul_rn(pg, aS[t * DP + c]);
                    gam[t] = pg;
                }
            }
            const bool fast = __syncthreads_and(gam[C - 1] >= 1e-30f);
            if (fast) {
                // the cumulative decays in place of alpha; then thread (t = tid % C, channels
                // 8 (tid / C) .. + 7) forms Khat, Qhat, Kchk and Ktil^T with 16-byte accesses
                // (a quarter warp covers 8 rows: no bank conflicts)
                if (hf == 0) {
#pragma unroll
                    for (int t = 0; t < C; ++t) aS[t * DP + c] = gam[t];
                    gC[c] = gam[C - 1];
                }
                __syncthreads();
                const int t = tid % C, c8 = 8 * (tid / C);
#pragma unroll
                for (int half4 = 0; half4 < 2; ++half4) {
                    const int cb = c8 + 4 * half4;
                    const float4 k4 = *reinterpret_cast<const float4 *>(kS + t * DP + cb);
                    const float4 q4 = *reinterpret_cast<const float4 *>(qS + t * DP + cb);
                    const float4 g4 = *reinterpret_cast<const float4 *>(aS + t * DP + cb);
                    const float4 gc4 = *reinterpret_cast<const float4 *>(gC + cb);
                    const float4 kh = make_float4(__fmul_rn(k4.x, g4.x), __fmul_rn(k4.y, g4.y), __fmul_rn(k4.z, g4.z),
                                                  __fmul_rn(k4.w, g4.w));
                    const float4 qh = make_float4(__fmul_rn(q4.x, g4.x), __fmul_rn(q4.y, g4.y), __fmul_rn(q4.z, g4.z),
                                                  __fmul_rn(q4.w, g4.w));
                    const float4 kc = make_float4(__fmul_rn(k4.x, __frcp_rn(g4.x)), __fmul_rn(k4.y, __frcp_rn(g4.y)),
                                                  __fmul_rn(k4.z, __frcp_rn(g4.z)), __fmul_rn(k4.w, __frcp_rn(g4.w)));
                    put_split4(smem + oB1h, smem + oB1l, tc::kmajor_offset(t, cb, D), kh.x, kh.y, kh.z, kh.w);
                    put_split4(smem + oB1h, smem + oB1l, tc::kmajor_offset(C + t, cb, D), qh.x, qh.y, qh.z, qh.w);
                    put_split(smem + oKTh, smem + oKTl, tc::kmajor_offset(cb, t, C), __fmul_rn(kc.x, gc4.x));
                    put_split(smem + oKTh, smem + oKTl, tc::kmajor_offset(cb + 1, t, C), __fmul_rn(kc.y, gc4.y));
                    put_split(smem + oKTh, smem + oKTl, tc::kmajor_offset(cb + 2, t, C), __fmul_rn(kc.z, gc4.z));
                    put_split(smem + oKTh, smem + oKTl, tc::kmajor_offset(cb + 3, t, C), __fmul_rn(kc.w, gc4.w));
                    *reinterpret_cast<float4 *>(kS + t * DP + cb) = kh;
                    *reinterpret_cast<float4 *>(qS + t * DP + cb) = qh;
                    *reinterpret_cast<float4 *>(aS + t * DP + cb) = kc;
                }
            } else if (hf == 0) {  // tiny decays: Khat rows, Ktil^T row c by running products
#pragma unroll
                for (int t = 0; t < C; ++t)
                    put_split(smem + oB1h, smem + oB1l, tc::kmajor_offset(t, c, D), __fmul_rn(kS[t * DP + c], gam[t]));
                float tail = 1.0f;  // prod_{s=i+1..C-1} alpha_s[c]
#pragma unroll
                for (int i = C - 1; i >= 0; --i) {
                    put_split(smem + oKTh, smem + oKTl, tc::kmajor_offset(c, i, C), __fmul_rn(kS[i * DP + c], tail));
                    tail = __fmul_rn(tail, aS[i * DP + c]);
                }
                gC[c] = gam[C - 1];
            } else {  // tiny decays: Qhat rows
#pragma unroll
                for (int t = 0; t < C; ++t)
                    put_split(smem + oB1h, smem + oB1l, tc::kmajor_offset(C + t, c, D), __fmul_rn(qS[t * DP + c], gam[t]));
            }
            __syncthreads();  // Gamma_C of every channel
            // ---- S0^T (hi, lo) as the A operand, Gamma_C S0^T as MMA 4's accumulator:
            // thread (v, hf) takes key channels 64 hf .. 64 hf + 63 of column v
            {
                const int ub = 64 * hf;
                float x[64];
                if (t0 == 0) {  // the staged copy ([u][v] row-major in the lo buffer)
                    const bool ok = mbar_wait_bounded(&bars[3], sph) || mbar_wait_bounded(&bars[3], sph);
                    if (!__syncthreads_and(ok)) {
                        failed = true;
                        break;
                    }
                    const float *st = reinterpret_cast<const float *>(smem + oSAl);
#pragma unroll
                    for (int u = 0; u < 64; ++u) x[u] = st[(ub + u) * D + v];
                    sph ^= 1u;
                    __syncthreads();  // every column read before the operands overwrite the copy
                } else {
#pragma unroll
                    for (int u0 = 0; u0 < 64; u0 += 16) {
                        float y[16];
                        tc::ld16(tm + cS + ub + u0, y);
#pragma unroll
                        for (int j = 0; j < 16; ++j) x[u0 + j] = y[j];
                    }
                    tc::wait_ld();
                }
#pragma unroll
                for (int u0 = 0; u0 < 64; u0 += 16) {
                    float y[16];
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        put_split4(smem + oSAh, smem + oSAl, tc::kmajor_offset(v, ub + u0 + j, D), x[u0 + j],
                                   x[u0 + j + 1], x[u0 + j + 2], x[u0 + j + 3]);
#pragma unroll
                    for (int j = 0; j < 16; ++j) y[j] = __fmul_rn(x[u0 + j], gC[ub + u0 + j]);
                    tc::st16(tm + cS + ub + u0, y);
                }
                tc::wait_st();
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            // ---- MMA 1: [P^T | Oq^T] = S0^T [Khat ; Qhat]^T
            if (tid == 0) {
                tc::fence_after_sync();
                const uint32_t id = tc::idesc_tf32(128, 2 * C);
#pragma unroll 1
                for (int s = 0; s < D / 8; ++s) {
                    const uint64_t ah = dSAh + 16 * s, al = dSAl + 16 * s;
                    const uint64_t bh = dB1h + 16 * s, bl = dB1l + 16 * s;
                    tc::mma_tf32(*tslot + cP, ah, bh, id, s > 0);
                    tc::mma_tf32(*tslot + cP, ah, bl, id, true);
                    tc::mma_tf32(*tslot + cP, al, bh, id, true);
                }
                tc::commit(&bars[0]);
            }
            // ---- meanwhile: A (scaled by beta) and Bm
            {
                const int e = tid;  // the parts above and on the diagonal that are zero
                const int te = e / C, ie = e - te * C;
                if (ie >= te) mA[te * C + ie] = 0.0f;
                if (ie > te) mB[te * C + ie] = 0.0f;
            }
            if (fast) {
                // pair p = (t, i), i <= t, in row order; thread pair (2p, 2p + 1) splits the
                // channels.  Every lane runs both rounds (the shuffles need the whole warp);
                // a lane without a pair in a round computes nothing and writes nothing.
                constexpr int kPairs = C * (C + 1) / 2;
#pragma unroll 1
                for (int round = 0; round < (kPairs + kThreads / 2 - 1) / (kThreads / 2); ++round) {
                    const int p = (tid >> 1) + round * (kThreads / 2);
                    const bool active = p < kPairs;
                    int t = 0;
                    while (active && (t + 1) * (t + 2) / 2 <= p) ++t;
                    const int i = active ? p - t * (t + 1) / 2 : 0;
                    float da = 0.0f, db = 0.0f;
                    if (active) {
                        const int c0 = 64 * (tid & 1);
                        const float4 *kt4 = reinterpret_cast<const float4 *>(kS + t * DP + c0);
                        const float4 *qt4 = reinterpret_cast<const float4 *>(qS + t * DP + c0);
                        const float4 *ki4 = reinterpret_cast<const float4 *>(aS + i * DP + c0);
#pragma unroll 4
                        for (int m = 0; m < 16; ++m) {
                            const float4 a4 = kt4[m], q4 = qt4[m], k4 = ki4[m];
                            da = __fmaf_rn(a4.x, k4.x, da);
                            da = __fmaf_rn(a4.y, k4.y, da);
                            da = __fmaf_rn(a4.z, k4.z, da);
                            da = __fmaf_rn(a4.w, k4.w, da);
                            db = __fmaf_rn(q4.x, k4.x, db);
                            db = __fmaf_rn(q4.y, k4.y, db);
                            db = __fmaf_rn(q4.z, k4.z, db);
                            db = __fmaf_rn(q4.w, k4.w, db);
                        }
                    }
                    da = __fadd_rn(da, __shfl_xor_sync(0xffffffffu, da, 1));
                    db = __fadd_rn(db, __shfl_xor_sync(0xffffffffu, db, 1));
                    if (active && (tid & 1) == 0) {
                        if (i < t) mA[t * C + i] = __fmul_rn(betaS[t], da);
                        mB[t * C + i] = db;
                    }
                }
            } else {
                // running products: thread (i, cq) takes channels cq + 16 m of row i
                const int i = tid >> 4, cq = tid & 15;
                float accA[C], accB[C];
#pragma unroll
                for (int t = 0; t < C; ++t) accA[t] = accB[t] = 0.0f;
#pragma unroll 1
                for (int m = 0; m < D / 16; ++m) {
                    const int cc = cq + 16 * m;
                    const float ki = kS[i * DP + cc];
                    float rho = 1.0f;  // prod_{s=i+1..t} alpha_s[cc]
#pragma unroll
                    for (int t = 0; t < C; ++t) {
                        if (t > i) rho = __fmul_rn(rho, aS[t * DP + cc]);
                        const float kr = __fmul_rn(ki, rho);
                        if (t > i) accA[t] = __fmaf_rn(kS[t * DP + cc], kr, accA[t]);
                        if (t >= i) accB[t] = __fmaf_rn(qS[t * DP + cc], kr, accB[t]);
                    }
                }
#pragma unroll
                for (int t = 0; t < C; ++t) {
#pragma unroll
                    for (int s = 1; s < 16; s <<= 1) {
                        accA[t] = __fadd_rn(accA[t], __shfl_xor_sync(0xffffffffu, accA[t], s));
                        accB[t] = __fadd_rn(accB[t], __shfl_xor_sync(0xffffffffu, accB[t], s));
                    }
                }
                if (cq == 0) {
#pragma unroll
                    for (int t = 0; t < C; ++t) {
                        if (t > i) mA[t * C + i] = __fmul_rn(betaS[t], accA[t]);
                        if (t >= i) mB[t * C + i] = accB[t];
                    }
                }
            }
            __syncthreads();
            {  // T = (I + L)^{-1} = (I - L)(I + L^2)(I + L^4)(I + L^8), L = diag(beta) A strictly
               // lower (L^16 = 0); thread tid owns entry (r, cc); scratch in the R/W buffer
                const int r = tid / C, cc = tid % C;
                float *Tc = reinterpret_cast<float *>(smem + oA2h);
                float *Pw = Tc + C * C, *Pn = Pw + C * C;
                Tc[tid] = (r == cc ? 1.0f : 0.0f) - mA[tid];
                Pw[tid] = mA[tid];
#pragma unroll 1
                for (int k = 0; k < 3; ++k) {
                    __syncthreads();
                    float acc = 0.0f;
#pragma unroll
                    for (int i2 = 0; i2 < C; ++i2) acc = __fmaf_rn(Pw[r * C + i2], Pw[i2 * C + cc], acc);
                    Pn[tid] = acc;  // L^(2^(k+1))
                    __syncthreads();
                    float t2 = Tc[tid];
#pragma unroll
                    for (int i2 = 0; i2 < C; ++i2) t2 = __fmaf_rn(Tc[r * C + i2], Pn[i2 * C + cc], t2);
                    __syncthreads();  // every thread has read Tc and Pw of this step
                    Tc[tid] = t2;
                    Pw[tid] = Pn[tid];
                }
                put_split(smem + oTh, smem + oTl, tc::kmajor_offset(r, cc, C), Tc[tid]);
            }
            put_split(smem + oBh, smem + oBl, tc::kmajor_offset(tid / C, tid % C, C), mB[tid]);  // C * C == kThreads
            fence_proxy_async_smem();
            // ---- MMA 1 done: R^T = diag(beta) (V^T - P^T) for tokens 8 hf .. 8 hf + 7
            if (!wait(0)) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            // the operand buffers are free: the next tile's state comes in now, and the
            // next group's inputs are fetched while this group finishes
            if (t0 + C < n) {
                fetch(item, t0 + C);
            } else {
                const bool nx_ok = nx_slot >= 0 && (int64_t)nx_slot < P.n_slots && nx_n >= 1 && nx_n <= L;
                staged = nx_ok ? nxi : next_work(nxi);
                prefetch_state(staged);
                if (staged < items) fetch(staged, 0);
            }
            {
                float pv[C], r[C / 2];
                tc::ld16(tm + cP, pv);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < C / 2; ++j) {
                    const int t = (C / 2) * hf + j;
                    r[j] = __fmul_rn(betaS[t], __fsub_rn(vt[j], hf ? pv[C / 2 + j] : pv[j]));
                }
#pragma unroll
                for (int j = 0; j < C / 2; j += 4)
                    put_split4(smem + oA2h, smem + oA2l, tc::kmajor_offset(v, (C / 2) * hf + j, C), r[j], r[j + 1],
                               r[j + 2], r[j + 3]);
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            // ---- MMA 2: W^T = R^T T^T
            if (tid == 0) {
                tc::fence_after_sync();
                const uint32_t id = tc::idesc_tf32(128, C);
#pragma unroll
                for (int s = 0; s < C / 8; ++s) {
                    const uint64_t ah = dA2h + 16 * s, al = dA2l + 16 * s;
                    const uint64_t bh = dTh + 16 * s, bl = dTl + 16 * s;
                    tc::mma_tf32(*tslot + cW, ah, bh, id, s > 0);
                    tc::mma_tf32(*tslot + cW, ah, bl, id, true);
                    tc::mma_tf32(*tslot + cW, al, bh, id, true);
                }
                tc::commit(&bars[1]);
            }
            if (!wait(1)) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            {
                float wv[C];
                tc::ld16(tm + cW, wv);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < C / 2; j += 4) {
                    const int t = (C / 2) * hf + j;
                    put_split4(smem + oA2h, smem + oA2l, tc::kmajor_offset(v, t, C),
                               hf ? wv[C / 2 + j] : wv[j], hf ? wv[C / 2 + j + 1] : wv[j + 1],
                               hf ? wv[C / 2 + j + 2] : wv[j + 2], hf ? wv[C / 2 + j + 3] : wv[j + 3]);
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            // ---- MMA 3: O^T = Oq^T + W^T Bm^T;  MMA 4: S_C^T = Gamma_C S0^T + W^T Ktil
            if (tid == 0) {
                tc::fence_after_sync();
                const uint32_t id16 = tc::idesc_tf32(128, C), id128 = tc::idesc_tf32(128, D);
#pragma unroll
                for (int s = 0; s < C / 8; ++s) {
                    const uint64_t ah = dA2h + 16 * s, al = dA2l + 16 * s;
                    const uint64_t bh = dBh + 16 * s, bl = dBl + 16 * s;
                    tc::mma_tf32(*tslot + cOq, ah, bh, id16, true);
                    tc::mma_tf32(*tslot + cOq, ah, bl, id16, true);
                    tc::mma_tf32(*tslot + cOq, al, bh, id16, true);
                    const uint64_t kh = dKTh + 16 * s, kl = dKTl + 16 * s;
                    tc::mma_tf32(*tslot + cS, ah, kh, id128, true);
                    tc::mma_tf32(*tslot + cS, ah, kl, id128, true);
                    tc::mma_tf32(*tslot + cS, al, kh, id128, true);
                }
                tc::commit(&bars[2]);
            }
            if (!wait(2)) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            if (o_g) {
                float ov[C];
                tc::ld16(tm + cOq, ov);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < C / 2; ++j) {
                    const int t = (C / 2) * hf + j;
                    if (t < nt)
                        store_from_f32<TO>(o_g + (((size_t)b * L + t0 + t) * Hv + h) * D + v,
                                           hf ? ov[C / 2 + j] : ov[j]);
                }
            }
            ph ^= 1u;
        }
        if (failed) break;
        // ---- the tile's final state back to HBM (thread (v, hf): key channels 64 hf ..)
#pragma unroll
        for (int u0 = 0; u0 < 64; u0 += 16) {
            float y[16];
            tc::ld16(tm + cS + 64 * hf + u0, y);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) Sg[(size_t)(64 * hf + u0 + j) * D + v] = y[j];
        }
        __syncthreads();  // the next tile restages the inputs
    }
    if (failed && tid == 0) report_bits(P.status, RS_DEV_PIPE_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (w == 0) tc::tmem_dealloc(*tslot, kTmemCols);
}

template <bool KDA, typename TI, typename TO>
cudaError_t run(PrefillParams &P, cudaStream_t s) {
    auto kern = chunk_prefill_kernel<KDA, TI, TO>;
    cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), kSmem);
    if (e != cudaSuccess) return e;
    const int items = P.B * P.Hv;
    int grid = device_sm_count();
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmem, s, P);
}

template <bool KDA>
cudaError_t by_types(const StepLaunch &L, PrefillParams &P, cudaStream_t s) {
    if (L.in_dt == RS_BF16 && L.out_dt == RS_F32) return run<KDA, __nv_bfloat16, float>(P, s);
    if (L.in_dt == RS_BF16 && L.out_dt == RS_BF16) return run<KDA, __nv_bfloat16, __nv_bfloat16>(P, s);
    if (L.in_dt == RS_F32 && L.out_dt == RS_F32) return run<KDA, float, float>(P, s);
    if (L.in_dt == RS_F16 && L.out_dt == RS_F32) return run<KDA, __half, float>(P, s);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_prefill_chunked(const StepLaunch &L, PrefillParams &P, cudaStream_t s) {
    if (L.D != 128 || L.khi >= 0) return cudaErrorNotSupported;  // FP32 layout, dk = dv = 128
    return L.kda ? by_types<true>(L, P, s) : by_types<false>(L, P, s);
}

}  // namespace rs
