// rs_chunk.cuh -- prefill chunks in the chunk-parallel form on the tensor
// cores (sm_103a; the FP32 state layout, and the mixed FP16/INT8 layouts --
// one INT8 scale per row, or DAMP-exact groups of 32 with value scaling --
// dequantised at a tile's start and requantised once at its end).
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
// lane v of every M = 128 product below (each takes half of the column's key
// channels or tokens).  The state lives in tensor memory as S^T (lane v,
// columns u) across the groups of a tile.  Per group of C = 32 tokens:
//   G       [Khat ; Qhat] Kchk^T  (the C x C matrices A and Bm)   (K = 128)
//   MMA 1   [P^T | Oq^T] = S0^T [Khat ; Qhat]^T      (K = 128, A in tensor memory)
//   MMA 2   W^T = R^T T^T, T = (I + diag(beta) A)^{-1}  (K = C)
//   MMA 3   O^T = Oq^T + W^T Bm^T                      (K = C)
//   MMA 4   S_C^T = Gamma_C S0^T + W^T Ktil             (K = C, N = 128)
// all of kind::tf32, which reads an fp32 operand as tf32 by dropping its low
// 13 mantissa bits: each operand x is taken as hi = x (so read) plus the
// exact remainder lo = x - hi, and the products hi*hi + hi*lo + lo*hi (about
// 2^-21 relative) accumulate in fp32 in tensor memory.  Where one operand is
// shared, its hi and lo parts stack along M or N so that one instruction
// makes two of the three products (G: [hi ; lo] rows of Khat and Qhat along
// M and of Kchk along N, all four products in one instruction; MMA 1 to 3:
// [hi ; lo] rows of the B operand), and the accumulator columns that hold
// them are summed when read.  A[t][i] = Khat_t . Kchk_i and
// Bm[t][i] = Qhat_t . Kchk_i with Kchk_i = k_i / Gamma_i (the decay products
// factor through the cumulative decay), unless some cumulative decay of the
// group falls below 1e-20, where the CUDA cores take the running product of
// each pair's decays instead; T by forward substitution through the unit
// lower triangular I + diag(beta) A.  In the factored form MMA 4 adds
// W^T Kchk to the unscaled S0^T and the decay Gamma_C is applied when the
// state is next read (the next group, or the tile's end): the same sum, with
// Ktil = Gamma_C Kchk, whose rounding is relative to the result either way.
// One thread issues a tensor-core instruction only about every hundred
// cycles, so the instructions of G, MMA 1 and MMA 2 come from several warps
// at once, each accumulating into tensor-memory columns of its own that are
// free at that moment; the parts are summed in a fixed order when read.
// A tile's state (64 KB FP32, or its packed tile) arrives by a bulk copy
// during the previous tile, each group's token vectors by tensor copies
// during the previous group, a full group's outputs leave by one tensor
// copy, and the final FP32 state by a bulk copy while the next tile starts
// (a packed tile is requantised from shared memory and its words stored by
// every thread).  On the DAMP-exact layout the state is T = S diag(c')^{-1}:
// the values enter as v / c' and the outputs leave as c' o.  The result
// equals the token-by-token recurrence up to rounding (not bit for bit: the
// order of the sums differs), and is the same on every call.
#pragma once

#include <cuda.h>  // CUtensorMap and the tiled-encode signature (called through the runtime)

#include <cstring>
#include <type_traits>

#include "rs_internal.h"
#include "rs_damp.h"
#include "rs_device.cuh"
#include "rs_step.cuh"  // the mixed layout's quantiser (quant_quad*) and its constants
#include "rs_tc.cuh"
#include "../../include/recurrent_state.h"

namespace rs {

namespace {

__device__ __forceinline__ void report_bits(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

constexpr int D = 128;                 // dk = dv
constexpr int C = 32;                  // tokens per group
constexpr int kThreads = 256;          // two threads per value column
constexpr uint32_t kTmemCols = 512;
constexpr int DP = D + 4;              // padded fp32 row of alpha / Gamma / Kchk (bank spread)

// shared memory (bytes): tf32 operands in the K-major core-matrix layout of
// rs_tc.cuh, hi and lo parts; the group's token vectors as copied in (rows of
// D values and 16 bytes of zeros, so that 16-byte reads by token stay clear of
// bank conflicts); small matrices
constexpr int kB1 = 2 * C * D * 4;     // [Khat ; Qhat] (N = 2C, K = u), per part
constexpr int kCC = C * C * 4;         // T or Bm (N = t, K = i)
constexpr int CA = C + 1;              // row of L = diag(beta) A in shared memory (bank spread)
constexpr int kKT = D * C * 4;         // Ktil^T (N = c, K = i)
constexpr int kA2 = D * C * 4;         // R^T, then W^T (M = v, K = t)
constexpr int kTok = C * DP * 4;       // [t][c] fp32 rows, or one token vector of the widest input type
constexpr int oB1h = 0, oB1l = oB1h + kB1;                   // also: the next tile's incoming state
constexpr int oKTh = oB1l + kB1, oKTl = oKTh + kKT;          // KT, A2: also a tile's final state and a
                                                             // packed tile's dequantised rows
constexpr int oA2h = oKTl + kKT, oA2l = oA2h + kA2;
constexpr int oTh = oA2l + kA2, oTl = oTh + kCC, oBh = oTl + kCC, oBl = oBh + kCC;  // also: a group's outputs
constexpr int oK = oBl + kCC, oQ = oK + kTok, oAl = oQ + kTok;
constexpr int oBeta = oAl + kTok, oAlpS = oBeta + C * 4, oGc = oAlpS + C * 4;
constexpr int oMA = oGc + D * 4;
constexpr int kBars = 7;
constexpr int oBar = oMA + C * CA * 4, oTslot = oBar + kBars * 8;
// the Gram products' B operand Kchk (N = i, K = c; hi and lo parts, 16 KB each) over the k and
// q rows, which the factored form no longer reads once Khat, Qhat and Kchk are formed
constexpr int oKCh = oK, oKCl = oK + C * D * 4;
static_assert(oKCl + C * D * 4 <= oAl, "Kchk operand fits the k and q rows");
constexpr int oV = (oTslot + 16 + 127) / 128 * 128;  // the group's v rows
// mixed layout: key channel -> physical row of the tile's head and the reverse map, the
// requantisation's row scales, their negations and reciprocals (by physical row), and the
// non-finite flag (DAMP-exact tiles: one scale per group of 32 columns, [group][row]; and the
// value-scaling factors)
constexpr int NGM = D / kDampGroup;
constexpr int oPinv = oV + kTok, oPiS = oPinv + D, oQs = oPiS + D, oQns = oQs + NGM * D * 4, oQrc = oQns + NGM * D * 4,
              oQflag = oQrc + NGM * D * 4, oCs = oQflag + 16;
constexpr int kSmem = oCs + D * 4;
constexpr int KHM = 16;  // FP16 rows of the mixed layout the chunked form takes
constexpr int kMixBytes = 2 * KHM * D + (D - KHM) * D + 4 * (D - KHM);  // 18,880 B
constexpr int kDampBytes = 2 * KHM * D + (D - KHM) * D + 4 * (D - KHM) * NGM;  // 20,224 B
static_assert(kMixBytes % 16 == 0 && kDampBytes % 16 == 0 && kDampBytes <= 2 * kB1,
              "a packed tile fits the staging buffers");
static_assert(kSmem <= 232448, "fits the shared memory of one SM");
static_assert(oKTh + D * D * 4 == oTh, "the final state fills KT and the R/W operand");
static_assert(2 * kB1 == D * D * 4, "a tile's incoming state fills the [Khat ; Qhat] operand buffers");
static_assert(oTl == oTh + kCC && oBl == oBh + kCC, "T and Bm: remainder rows follow the high rows");
static_assert(oBar % 8 == 0 && oKTh % 16 == 0 && oA2h % 16 == 0, "alignment");
static_assert(oK % 128 == 0 && oAl % 128 == 0 && oV % 128 == 0, "tensor-copy destinations");

// The group's token vectors come in by 3-D tensor copies: a tensor [rows][heads][D]
// (rows = sequence x token) and a box of C rows of one head, D + 16 bytes wide
// (the columns past D lie outside the tensor and arrive as zeros).
struct ChunkMaps {
    CUtensorMap k, q, v, a;  // a: per-channel decays (KDA)
    CUtensorMap o;           // the outputs, box of C rows by D (used when o_rows != 0)
    int o_rows;              // 1: a full group's outputs leave by one tensor copy
};
// C rows of one head from shared memory to a [rows][heads][D] tensor (a bulk group of this thread)
__device__ __forceinline__ void tma_store_rows(const CUtensorMap *map, const void *src, int head, int row) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(0), "r"(head), "r"(row), "r"(smem_addr(src))
        : "memory");
}
__device__ __forceinline__ void tma_rows(void *dst, const CUtensorMap *map, int head, int row, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(head), "r"(row), "r"(smem_addr(bar))
        : "memory");
}
// 16 consecutive input values (16-byte aligned) as fp32
template <typename TI>
__device__ __forceinline__ void load16(const uint8_t *p, float (&x)[16]) {
    if constexpr (sizeof(TI) == 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 f = reinterpret_cast<const float4 *>(p)[j];
            x[4 * j] = f.x, x[4 * j + 1] = f.y, x[4 * j + 2] = f.z, x[4 * j + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint4 u = reinterpret_cast<const uint4 *>(p)[j];
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * j + 2 * e] = load_as_f32<TI>(reinterpret_cast<const TI *>(&wd[e]));
                x[8 * j + 2 * e + 1] = load_as_f32<TI>(reinterpret_cast<const TI *>(&wd[e]) + 1);
            }
        }
    }
}

// tensor-memory columns: S^T (also MMA 1's high part) and its remainder; MMA 1's accumulator
// D1 = [hi*hi + lo*hi of P^T | of Oq^T | hi*lo of P^T | of Oq^T]; the Gram products G (Kchk's high
// parts | remainders); W^T
// (MMA 2: [hi*hi + lo*hi | hi*lo]), whose columns then take MMA 3's W^T Bm^T likewise
constexpr uint32_t cS = 0, cSl = D, cD1 = 2 * D, cG = 3 * D, cW = 3 * D + 2 * C;
static_assert(cW + 2 * C <= kTmemCols, "tensor memory");
constexpr float kFastMin = 1e-20f;  // smallest cumulative decay of the factored form

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
// 1 / x by the hardware's approximate reciprocal (about 1 ulp; x a normal number here): Kchk only enters
// products held to the FP32 state's tolerance, so a correctly rounded quotient is not needed
__device__ __forceinline__ float rcp_fast(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
    return make_float4(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y), __fmul_rn(a.z, b.z), __fmul_rn(a.w, b.w));
}

// MIX: the pool holds mixed FP16/INT8 tiles (16 FP16 rows, one INT8 scale per row, row map pi);
// GRP: DAMP-exact ones (INT8 scales per group of 32 columns, value scaling c': the state is
// T = S diag(c')^{-1}, the values v' = v / c' and the outputs c' o'; PT carries c');
// FUSED: their requantisation arithmetic is the fused one
template <bool KDA, bool MIX, bool GRP, bool FUSED, typename TI, typename TO, typename PT>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_prefill_kernel(const __grid_constant__ PT P, const __grid_constant__ ChunkMaps M) {
    static_assert(MIX || !GRP, "DAMP-exact tiles are mixed tiles");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, w = tid >> 5;
    const int v = tid & (D - 1);  // value column (and key channel c in the per-channel work)
    const int hf = tid >> 7;      // which half of the column's channels / tokens
    // the group's vectors as copied in: k and q rows (then the Kchk operand), v rows; alpha
    // rows (KDA) land in aS, which then holds Gamma and Kchk
    constexpr int RP = D * (int)sizeof(TI) + 16;  // bytes per copied row
    static_assert(2 * C * RP <= 2 * kTok && C * RP <= kTok, "copied rows fit");
    const uint8_t *rawK = smem + oK, *rawQ = smem + oK + C * RP, *rawV = smem + oV;
    float *aS = reinterpret_cast<float *>(smem + oAl);  // [t][DP]: alpha, Gamma, then Kchk
    float *betaS = reinterpret_cast<float *>(smem + oBeta);
    float *alpS = reinterpret_cast<float *>(smem + oAlpS);
    float *gC = reinterpret_cast<float *>(smem + oGc);
    float *mA = reinterpret_cast<float *>(smem + oMA);  // L = diag(beta) A, row stride CA
    // mbarriers: MMA 1, MMA 2, MMA 3, state copy, input copy, Gram, MMA 4 (the Gram products are
    // issued by four warps, MMA 1 and MMA 2 by two, each committing once)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + oBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + oTslot);

    if (tid == 0)
        for (int i = 0; i < kBars; ++i) mbar_init(&bars[i], i == 5 ? 4 : i < 2 ? 2 : 1);
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
    const uint32_t tbase = *tslot;
    const uint32_t tm = tbase + ((uint32_t)(32 * (w & 3)) << 16);  // this warp's 32 lanes
    // Several warps issue tensor-core instructions at once (one thread issues one only about
    // every hundred cycles).  Each issuing thread accumulates into columns of its own, and the
    // parts are summed in a fixed order when read, so results do not depend on the order in
    // which the pipe takes the warps' instructions.
    // operand descriptors at k-step 0; step s is 256 s bytes on, i.e. + 16 s in the address field
    const uint64_t dB1h = tc::smem_desc(smem + oB1h, 128, D * 32), dB1l = tc::smem_desc(smem + oB1l, 128, D * 32);
    const uint64_t dA2h = tc::smem_desc(smem + oA2h, 128, C * 32), dA2l = tc::smem_desc(smem + oA2l, 128, C * 32);
    const uint64_t dTh = tc::smem_desc(smem + oTh, 128, C * 32), dTl = tc::smem_desc(smem + oTl, 128, C * 32);
    const uint64_t dBh = tc::smem_desc(smem + oBh, 128, C * 32), dBl = tc::smem_desc(smem + oBl, 128, C * 32);
    const uint64_t dKTh = tc::smem_desc(smem + oKTh, 128, C * 32), dKTl = tc::smem_desc(smem + oKTl, 128, C * 32);
    // the Gram products' A operand: [Khat ; Qhat] high parts (rows 0..63) then remainders (rows 64..127)
    const uint64_t dG = tc::smem_desc(smem + oB1h, 128, D * 32);
    const uint64_t dKCh = tc::smem_desc(smem + oKCh, 128, D * 32), dKCl = tc::smem_desc(smem + oKCl, 128, D * 32);
    // MMA 1: D1 = S0^T [Khat ; Qhat ; Khat_lo ; Qhat_lo]^T + S0_lo^T [Khat ; Qhat]^T, issued by one
    // thread of warp 2 (k-steps 0..7 of the 16, both terms, into the D1 columns) and of warp 3
    // (k-steps 8..15, into the Gram and W^T columns, then free); R and the outputs add the two parts
    auto issue_mma1 = [&]() {
        if ((tid & 31) == 0) {
            tc::fence_after_sync();
            const uint32_t i4 = tc::idesc_tf32(128, 4 * C), i2 = tc::idesc_tf32(128, 2 * C);
            const uint32_t acc = tbase + (w == 2 ? cD1 : cG);
            const int s0 = (w - 2) * (D / 16);
#pragma unroll 1
            for (int s = s0; s < s0 + D / 16; ++s) {
                tc::mma_tf32_ta(acc, tbase + cS + 8 * s, dB1h + 16 * s, i4, s > s0);
                tc::mma_tf32_ta(acc, tbase + cSl + 8 * s, dB1h + 16 * s, i2, true);
            }
            tc::commit(&bars[0]);
        }
    };

    const int Hv = P.Hv, Hk = P.Hk, L = P.L;
    constexpr int kStateBytes = MIX ? (GRP ? kDampBytes : kMixBytes) : D * D * 4;
    float *csS = reinterpret_cast<float *>(smem + oCs);  // DAMP-exact: c' of the tile's head
    uint8_t *pool = static_cast<uint8_t *>(P.pool);
    uint8_t *pinv = smem + oPinv;  // key channel -> physical row
    uint8_t *piS = smem + oPiS;    // physical row -> key channel
    const uint32_t *pi4 = reinterpret_cast<const uint32_t *>(piS);  // the key channels of four physical rows
    const int items = P.B * Hv;
    TO *o_g = static_cast<TO *>(P.o);
    uint32_t ph = 0, sph = 0, iph = 0, gph = 0;  // barrier parities: MMAs, state copy, input copy, Gram
    bool failed = false;
    // the barriers with copies or MMAs in flight (bit k: bars[k]; the same in every thread)
    uint32_t pendm = 0;

    auto wait_bar = [&](int k, uint32_t parity) -> bool {
        const bool ok = mbar_wait_bounded(&bars[k], parity) || mbar_wait_bounded(&bars[k], parity);
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
    // a group's token vectors by tensor copies (thread `issuer` issues them), the per-token scalars
    // (beta, GDN alpha) into registers of threads 0..C-1; rows past the sequence's tokens are
    // copied too and masked where read
    constexpr uint32_t kInBytes = 3u * C * RP + (KDA ? (uint32_t)C * DP * 4 : 0u);
    float fb = 0.0f, fga = 1.0f;  // beta and the GDN decay of token tid of the fetched group
    auto fetch = [&](int it, int tb, int nn, int issuer) {  // nn: the sequence's token count
        const int bb = it / Hv, hh = it - bb * Hv, gg = hh / (Hv / Hk);
        const int ntt = min(C, nn - tb);
        if (tid == issuer) {
            const int row = bb * L + tb;
            mbar_arrive_expect_tx(&bars[4], kInBytes);
            tma_rows(smem + oK, &M.k, gg, row, &bars[4]);
            tma_rows(smem + oK + C * RP, &M.q, gg, row, &bars[4]);
            tma_rows(smem + oV, &M.v, hh, row, &bars[4]);
            if (KDA) tma_rows(smem + oAl, &M.a, hh, row, &bars[4]);
        }
        pendm |= 1u << 4;
        fb = 0.0f, fga = 1.0f;
        if (tid < ntt) {
            const size_t bt = (size_t)bb * L + tb + tid;
            fb = P.beta[bt * Hv + hh];
            if (!KDA) fga = P.alpha[bt * Hv + hh];
        }
    };
    // a tile's state by bulk copies into the [Khat ; Qhat] operand buffers, free from the end of
    // the previous tile's last MMA 1 until this tile's first group has read them
    auto load_state = [&](int it) {
        const int bb = it / Hv, hh = it - bb * Hv;
        const uint8_t *src = pool + ((size_t)P.slot_idx[bb] * Hv + hh) * kStateBytes;
        if (tid == 0) {
            mbar_arrive_expect_tx(&bars[3], (uint32_t)kStateBytes);
            bulk_g2s(smem + oB1h, src, kStateBytes, &bars[3]);  // the whole tile in one copy
        }
        pendm |= 1u << 3;
    };
    {
        const int first = next_work(blockIdx.x);
        if (first < items) {
            load_state(first);
            fetch(first, 0, P.n_tokens ? P.n_tokens[first / Hv] : L, 0);
        }
    }
    // slot and token count of the current tile, read one tile ahead
    int32_t c_slot = -1, c_n = 0;
    if ((int)blockIdx.x < items) {
        c_slot = P.slot_idx[blockIdx.x / Hv];
        c_n = P.n_tokens ? P.n_tokens[blockIdx.x / Hv] : L;
    }
    // mixed layouts: thread tid < D holds pi[tid] of the current tile's head, read one tile ahead
    int c_pi = (MIX && tid < D && (int)blockIdx.x < items) ? P.pi[((int)blockIdx.x % Hv) * D + tid] : 0;

    for (int item = blockIdx.x; item < items && !failed; item += gridDim.x) {
        const int b = item / Hv, h = item - b * Hv;
        const int32_t slot = c_slot, n = c_n;
        const int nxi = item + gridDim.x;
        c_slot = nxi < items ? P.slot_idx[nxi / Hv] : -1;
        c_n = nxi < items ? (P.n_tokens ? P.n_tokens[nxi / Hv] : L) : 0;
        const int pi_t = c_pi;
        if (MIX && tid < D && nxi < items) c_pi = P.pi[(nxi % Hv) * D + tid];
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
        uint8_t *tile_g = pool + ((size_t)slot * Hv + h) * kStateBytes;
        float *Sg = reinterpret_cast<float *>(tile_g);
        if constexpr (GRP) {  // this head's value-scaling factors
            if (tid < D) csS[tid] = P.cs[h * D + tid];
        }
        // the next tile this CTA processes (its state and first vectors come in during this
        // tile's last group)
        const bool nx_ok = c_slot >= 0 && (int64_t)c_slot < P.n_slots && c_n >= 1 && c_n <= L;
        int nxt = items, nxt_n = 0;

        for (int t0 = 0; t0 < n && !failed; t0 += C) {
            const int nt = min(C, n - t0);
            const bool last = t0 + C >= n;
            // ---- the group's vectors (copied in during the previous group, or at start); pads
            // (t >= nt): k = q = v = 0, alpha = 1, beta = 0
            if (tid < C) {
                betaS[tid] = fb;
                alpS[tid] = fga;
            }
            if (!wait_bar(4, iph)) {
                failed = true;
                break;
            }
            iph ^= 1u;
            pendm &= ~(1u << 4);
            if (t0 == 0) {
                // this head's row map both ways (every thread has left the previous tile, whose
                // requantisation read them; the state-copy barrier orders them before use)
                if (MIX && tid < D) {
                    piS[tid] = (uint8_t)pi_t;
                    pinv[pi_t] = (uint8_t)tid;
                }
                if (!wait_bar(3, sph)) {
                    failed = true;
                    break;
                }
                sph ^= 1u;
                pendm &= ~(1u << 3);
                if constexpr (MIX) {
                    // the packed tile dequantised into FP32 rows of key-channel order in the staging
                    // buffers: thread (v, hf) takes column v of 18 of the 36 word rows (hf = 0: the 8
                    // FP16 pair rows and INT8 quads 0..9; hf = 1: quads 10..27) and writes physical
                    // row r to row pi[r]; each batch's loads go ahead of its stores
                    const uint8_t *stt = smem + oB1h;
                    float *stg = reinterpret_cast<float *>(smem + oKTh);
                    const uint32_t *hw = reinterpret_cast<const uint32_t *>(stt);
                    const uint32_t *lw = reinterpret_cast<const uint32_t *>(stt + 2 * KHM * D);
                    const float *sc = reinterpret_cast<const float *>(stt + 2 * KHM * D + (D - KHM) * D);
                    constexpr int kQuads = (D - KHM) / 4, kQB = 6;
                    auto quads = [&](int q0, int q1) {  // INT8 quads q0 .. q1 - 1
                        for (int b0 = q0; b0 < q1; b0 += kQB) {
                            uint32_t wd[kQB], pr[kQB];
                            float4 s4[kQB];
#pragma unroll
                            for (int i = 0; i < kQB; ++i) {
                                const int qd = min(b0 + i, q1 - 1);  // (a batch's tail repeats the last quad)
                                wd[i] = lw[qd * D + v];
                                pr[i] = pi4[KHM / 4 + qd];
                                // the scales of rows KHM + 4 qd .. + 3 (DAMP-exact: of column v's group)
                                s4[i] = GRP ? make_float4(sc[(4 * qd) * NGM + (v >> 5)], sc[(4 * qd + 1) * NGM + (v >> 5)],
                                                          sc[(4 * qd + 2) * NGM + (v >> 5)], sc[(4 * qd + 3) * NGM + (v >> 5)])
                                            : *reinterpret_cast<const float4 *>(sc + 4 * qd);
                            }
#pragma unroll
                            for (int i = 0; i < kQB; ++i) {
                                stg[(pr[i] & 0xffu) * D + v] = __fmul_rn((float)(int8_t)(wd[i] & 0xffu), s4[i].x);
                                stg[((pr[i] >> 8) & 0xffu) * D + v] = __fmul_rn((float)(int8_t)((wd[i] >> 8) & 0xffu), s4[i].y);
                                stg[((pr[i] >> 16) & 0xffu) * D + v] = __fmul_rn((float)(int8_t)((wd[i] >> 16) & 0xffu), s4[i].z);
                                stg[(pr[i] >> 24) * D + v] = __fmul_rn((float)(int8_t)(wd[i] >> 24), s4[i].w);
                            }
                        }
                    };
                    if (hf == 0) {
                        uint32_t wh[KHM / 2], ph[KHM / 4];
#pragma unroll
                        for (int j = 0; j < KHM / 2; ++j) wh[j] = hw[j * D + v];
#pragma unroll
                        for (int j = 0; j < KHM / 4; ++j) ph[j] = pi4[j];
#pragma unroll
                        for (int j = 0; j < KHM / 2; ++j) {  // FP16 rows 2 j, 2 j + 1
                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&wh[j]));
                            const uint32_t p2 = ph[j >> 1] >> (16 * (j & 1));
                            stg[(p2 & 0xffu) * D + v] = f.x;
                            stg[((p2 >> 8) & 0xffu) * D + v] = f.y;
                        }
                        quads(0, (kQuads - KHM / 2) / 2);
                    } else {
                        quads((kQuads - KHM / 2) / 2, kQuads);
                    }
                    __syncthreads();
                }
            }
            auto kv = [&](int t, int cc) -> float {  // k and q of token t, channel cc (0 for pads)
                return t < nt ? load_as_f32<TI>(reinterpret_cast<const TI *>(rawK + t * RP) + cc) : 0.0f;
            };
            auto qv = [&](int t, int cc) -> float {
                return t < nt ? load_as_f32<TI>(reinterpret_cast<const TI *>(rawQ + t * RP) + cc) : 0.0f;
            };
            // ---- S0^T and its tf32 remainder in tensor memory (MMA 1's A operand): thread (v, hf)
            // takes key channels 64 hf .. 64 hf + 63 of column v, from the staged copy (a tile's
            // first group) or from the state columns times the previous group's pending decay
#pragma unroll
            for (int u0 = 0; u0 < 64; u0 += 32) {
                const int ub = 64 * hf + u0;
                float x[16], x2[16], lo[16];
                if (t0 == 0) {  // the staged state (mixed: dequantised into the staging buffers)
                    const float *st = reinterpret_cast<const float *>(smem + (MIX ? oKTh : oB1h));
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        x[j] = st[(ub + j) * D + v];
                        x2[j] = st[(ub + 16 + j) * D + v];
                    }
                } else {
                    tc::ld16(tm + cS + ub, x);
                    tc::ld16(tm + cS + ub + 16, x2);
                    tc::wait_ld_regs(x, x2);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        x[j] = __fmul_rn(x[j], gC[ub + j]);
                        x2[j] = __fmul_rn(x2[j], gC[ub + 16 + j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) lo[j] = x[j] - tc::tf32_hi(x[j]);
                tc::st16(tm + cS + ub, x);
                tc::st16(tm + cSl + ub, lo);
#pragma unroll
                for (int j = 0; j < 16; ++j) lo[j] = x2[j] - tc::tf32_hi(x2[j]);
                tc::st16(tm + cS + ub + 16, x2);
                tc::st16(tm + cSl + ub + 16, lo);
            }
            tc::wait_st();
            tc::fence_before_sync();
            // ---- cumulative decays Gamma_t[c] of channel c = v; the factored form if none is tiny
            // (thread (c, 0) needs tokens 0..15 of the fast form, thread (c, 1) all of them)
            const int c = v;
            float gam[C];
            {
                float pg = 1.0f;
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    if (hf == 0 && t >= C / 2) break;
                    const float a = KDA ? (t < nt ? aS[t * DP + c] : 1.0f) : alpS[t];
                    pg = __fmul_rn(pg, a);
                    gam[t] = pg;
                }
            }
            // (also: every thread's state columns are written and the staged state and the
            // pending decays are read)
            const bool fast = __syncthreads_and(hf == 0 || gam[C - 1] >= kFastMin);
            if (fast) {
#pragma unroll
                for (int j = 0; j < C / 2; ++j) aS[((C / 2) * hf + j) * DP + c] = hf ? gam[C / 2 + j] : gam[j];
                if (hf == 1) gC[c] = gam[C - 1];
                __syncthreads();
                // thread (t = tid % C, channels 16 (tid / C) .. + 15): the Khat and Qhat operands
                // and Kchk (fp32 rows now, its operand once every k and q row has been read),
                // with 16-byte accesses (a quarter warp spans 8 rows)
                const int t = tid % C, cb0 = 16 * (tid / C);
                const bool real = t < nt;
                float kx[16], qx[16];
                load16<TI>(rawK + t * RP + cb0 * (int)sizeof(TI), kx);
                load16<TI>(rawQ + t * RP + cb0 * (int)sizeof(TI), qx);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int cb = cb0 + 4 * q4;
                    const float4 k4 = real ? make_float4(kx[4 * q4], kx[4 * q4 + 1], kx[4 * q4 + 2], kx[4 * q4 + 3])
                                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    const float4 qv4 = real ? make_float4(qx[4 * q4], qx[4 * q4 + 1], qx[4 * q4 + 2], qx[4 * q4 + 3])
                                            : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    const float4 g4 = *reinterpret_cast<const float4 *>(aS + t * DP + cb);
                    const float4 kh = mul4(k4, g4), qh = mul4(qv4, g4);
                    const float4 kc = make_float4(__fmul_rn(k4.x, rcp_fast(g4.x)), __fmul_rn(k4.y, rcp_fast(g4.y)),
                                                  __fmul_rn(k4.z, rcp_fast(g4.z)), __fmul_rn(k4.w, rcp_fast(g4.w)));
                    put_split4(smem + oB1h, smem + oB1l, tc::kmajor_offset(t, cb, D), kh.x, kh.y, kh.z, kh.w);
                    put_split4(smem + oB1h, smem + oB1l, tc::kmajor_offset(C + t, cb, D), qh.x, qh.y, qh.z, qh.w);
                    *reinterpret_cast<float4 *>(aS + t * DP + cb) = kc;
                }
            } else if (hf == 0) {  // tiny decays: Khat rows of channel c; alpha of the pads 1
                float pg = gam[C / 2 - 1];
#pragma unroll
                for (int t = C / 2; t < C; ++t) {
                    pg = __fmul_rn(pg, KDA ? (t < nt ? aS[t * DP + c] : 1.0f) : alpS[t]);
                    gam[t] = pg;
                }
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    put_split(smem + oB1h, smem + oB1l, tc::kmajor_offset(t, c, D), __fmul_rn(kv(t, c), gam[t]));
                    if (!KDA) aS[t * DP + c] = alpS[t];
                    else if (t >= nt) aS[t * DP + c] = 1.0f;
                }
                gC[c] = gam[C - 1];
            } else {  // tiny decays: Qhat rows of channel c
#pragma unroll
                for (int t = 0; t < C; ++t)
                    put_split(smem + oB1h, smem + oB1l, tc::kmajor_offset(C + t, c, D), __fmul_rn(qv(t, c), gam[t]));
            }
            __syncthreads();  // Gamma_C of every channel; every k and q row read
            if (fast) {
                const int t = tid % C, cb0 = 16 * (tid / C);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {  // this thread's own Kchk values
                    const float4 kc = *reinterpret_cast<const float4 *>(aS + t * DP + cb0 + 4 * q4);
                    put_split4(smem + oKCh, smem + oKCl, tc::kmajor_offset(t, cb0 + 4 * q4, D), kc.x, kc.y, kc.z, kc.w);
                }
            }
            if (tid == 0) bulk_store_wait_read();  // the previous tile's final state has left KT / A2
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();  // operands in place
            // ---- the Gram products (factored form): G = [Khat_hi ; Qhat_hi ; Khat_lo ; Qhat_lo]
            // [Kchk_hi ; Kchk_lo]^T, so that A = G[0..31] + G[64..95] and Bm = G[32..63] +
            // G[96..127] (each the sum of its two column halves) hold all four products of the
            // split pairs.  One thread in each of warps 0..3 issues a quarter of the k-steps into
            // 64 columns of its own (the MMA 1 and W^T columns are free until the parts are read);
            // MMA 1 waits until then, so that the Gram products have the pipe to themselves.
            if (fast && w < 4 && (tid & 31) == 0) {
                tc::fence_after_sync();
                // B = [Kchk_hi ; Kchk_lo] (64 rows): columns 0..31 of G take the high parts, 32..63 the
                // remainders
                const uint32_t ig = tc::idesc_tf32(128, 2 * C);
                const uint32_t acc = tbase + (w == 0 ? cG : w == 1 ? cW : cD1 + (w - 2) * 2 * C);
                const int s0 = w * (D / 32);
#pragma unroll 1
                for (int s = s0; s < s0 + D / 32; ++s) tc::mma_tf32(acc, dG + 16 * s, dKCh + 16 * s, ig, s > s0);
                tc::commit(&bars[5]);
            }
            if (fast) pendm |= 1u << 5;
            // ---- meanwhile: Ktil^T (factored form: Kchk^T, the decay pending), then
            // L = diag(beta) A, the Bm operand and T on the CUDA cores
            if (fast) {  // thread (c, i = 16 hf ..), 4 i per store
#pragma unroll
                for (int i0 = 0; i0 < C / 2; i0 += 4) {
                    const int i = (C / 2) * hf + i0;
                    put_split4(smem + oKTh, smem + oKTl, tc::kmajor_offset(v, i, C), aS[i * DP + v],
                               aS[(i + 1) * DP + v], aS[(i + 2) * DP + v], aS[(i + 3) * DP + v]);
                }
            } else if (hf == 0) {  // running products of the decays
                float tail = 1.0f;  // prod_{s=i+1..C-1} alpha_s[c]
#pragma unroll
                for (int i = C - 1; i >= 0; --i) {
                    put_split(smem + oKTh, smem + oKTl, tc::kmajor_offset(c, i, C), __fmul_rn(kv(i, c), tail));
                    tail = __fmul_rn(tail, aS[i * DP + c]);
                }
            }
            if (fast) {
                // G row m = lane v, columns i = 16 hf .. 16 hf + 15; the remainder rows (v >= 64)
                // pass through shared memory (the R/W buffer, free until R) to rows v - 64
                if (!wait_bar(5, gph)) {
                    failed = true;
                    break;
                }
                gph ^= 1u;
                pendm &= ~(1u << 5);
                tc::fence_after_sync();
                float g[16];
#pragma unroll
                for (int half = 0; half < 2; ++half) {  // the high-part columns, then the remainders'
                    const uint32_t off = half * C + (C / 2) * hf;
                    float a0[16], a1[16], a2[16], a3[16];
                    tc::ld16(tm + cG + off, a0);
                    tc::ld16(tm + cW + off, a1);
                    tc::ld16(tm + cD1 + off, a2);
                    tc::ld16(tm + cD1 + 2 * C + off, a3);
                    tc::wait_ld_regs(a0, a1);
                    tc::wait_ld_regs(a2, a3);
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) {
                        const float sj = __fadd_rn(__fadd_rn(__fadd_rn(a0[j], a1[j]), a2[j]), a3[j]);
                        g[j] = half ? __fadd_rn(g[j], sj) : sj;
                    }
                }
                float *G2 = reinterpret_cast<float *>(smem + oA2h);  // [64][CA]
                if (v >= 2 * C) {
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) G2[(v - 2 * C) * CA + (C / 2) * hf + j] = g[j];
                }
                tc::fence_before_sync();
                __syncthreads();  // the Gram parts are read: MMA 1 may overwrite them
                if (w == 2 || w == 3) {
                    issue_mma1();
                } else if (v < 2 * C) {
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) g[j] = __fadd_rn(g[j], G2[v * CA + (C / 2) * hf + j]);
                    if (v < C) {  // row t = v of A
                        const float bt = betaS[v];
#pragma unroll
                        for (int j = 0; j < C / 2; ++j) {
                            const int i = (C / 2) * hf + j;
                            if (i < v) mA[v * CA + i] = __fmul_rn(bt, g[j]);
                        }
                    } else {  // row t = v - C of Bm, zero above the diagonal
                        const int t = v - C;
#pragma unroll
                        for (int j = 0; j < C / 2; j += 4) {
                            const int i = (C / 2) * hf + j;
                            put_split4(smem + oBh, smem + oBl, tc::kmajor_offset(t, i, C), i <= t ? g[j] : 0.0f,
                                       i + 1 <= t ? g[j + 1] : 0.0f, i + 2 <= t ? g[j + 2] : 0.0f,
                                       i + 3 <= t ? g[j + 3] : 0.0f);
                        }
                    }
                }
            } else {
                // running products: thread (i, cq) takes channels cq + 8 m of row i
                const int i = tid >> 3, cq = tid & 7;
                float accA[C], accB[C];
#pragma unroll
                for (int t = 0; t < C; ++t) accA[t] = accB[t] = 0.0f;
#pragma unroll 1
                for (int m = 0; m < D / 8; ++m) {
                    const int cc = cq + 8 * m;
                    const float ki = kv(i, cc);
                    float rho = 1.0f;  // prod_{s=i+1..t} alpha_s[cc]
#pragma unroll
                    for (int t = 0; t < C; ++t) {
                        if (t > i) rho = __fmul_rn(rho, aS[t * DP + cc]);
                        const float kr = __fmul_rn(ki, rho);
                        if (t > i) accA[t] = __fmaf_rn(kv(t, cc), kr, accA[t]);
                        if (t >= i) accB[t] = __fmaf_rn(qv(t, cc), kr, accB[t]);
                    }
                }
#pragma unroll
                for (int t = 0; t < C; ++t) {
#pragma unroll
                    for (int s = 1; s < 8; s <<= 1) {
                        accA[t] = __fadd_rn(accA[t], __shfl_xor_sync(0xffffffffu, accA[t], s));
                        accB[t] = __fadd_rn(accB[t], __shfl_xor_sync(0xffffffffu, accB[t], s));
                    }
                }
                if (cq == 0) {
#pragma unroll
                    for (int t = 0; t < C; ++t) {
                        if (t > i) mA[t * CA + i] = __fmul_rn(betaS[t], accA[t]);
                        put_split(smem + oBh, smem + oBl, tc::kmajor_offset(t, i, C), t >= i ? accB[t] : 0.0f);
                    }
                }
            }
            if (fast) {  // warps 2 and 3 are issuing MMA 1; L and Bm are in place for the others
                if (w != 2 && w != 3) group_sync(1, kThreads - 64);
            } else {
                __syncthreads();
                if (w == 2 || w == 3) issue_mma1();
            }
            if (w >= 4) {
                // ---- T = (I + L)^{-1} by forward substitution, L = diag(beta) A strictly lower:
                // thread (column j = (tid - 128) / 4, r = tid % 4) of warps 4..7 holds T[r + 4 m][j],
                // m = 0..7, and takes T[i][j] from its owner by shuffle once row i is final
                const int j = (tid - kThreads / 2) >> 2, r = tid & 3;
                float x[8], lc[8], ln[8];  // L[r + 4 m][i] of this step and the next
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    x[m] = (r + 4 * m == j) ? 1.0f : 0.0f;
                    lc[m] = mA[(r + 4 * m) * CA];
                }
#pragma unroll
                for (int i = 0; i < C - 1; ++i) {
#pragma unroll
                    for (int m = 0; m < 8; ++m) ln[m] = i + 1 < C - 1 ? mA[(r + 4 * m) * CA + i + 1] : 0.0f;
                    const float xi = __shfl_sync(0xffffffffu, x[i >> 2], (tid & 28) | (i & 3));
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int t = r + 4 * m;
                        if (t > i) x[m] = __fmaf_rn(-lc[m], xi, x[m]);
                        lc[m] = ln[m];
                    }
                }
#pragma unroll
                for (int m = 0; m < 8; ++m)  // T as a B operand: row t, K = j
                    put_split(smem + oTh, smem + oTl, tc::kmajor_offset(r + 4 * m, j, C), x[m]);
            }
            pendm |= 1u;
            fence_proxy_async_smem();
            // ---- MMA 1 done
            if (!wait_bar(0, ph)) {
                failed = true;
                break;
            }
            pendm &= ~1u;
            tc::fence_after_sync();
            if (last) {  // the next tile's state into the operand buffers, free from here on
                nxt = nx_ok ? nxi : next_work(nxi);
                nxt_n = nxt >= items ? 0 : nxt == nxi ? c_n : (P.n_tokens ? P.n_tokens[nxt / Hv] : L);
                if (nxt < items) load_state(nxt);
            }
            if (!fast) {  // running products: MMA 4 adds Ktil^T W to Gamma_C S0^T, scaled now
#pragma unroll
                for (int u0 = 0; u0 < 64; u0 += 16) {
                    const int ub = 64 * hf + u0;
                    float x[16];
                    tc::ld16_wait(tm + cS + ub, x);
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] = __fmul_rn(x[j], gC[ub + j]);
                    tc::st16(tm + cS + ub, x);
                }
                tc::wait_st();
                tc::fence_before_sync();
            }
            // ---- R^T = diag(beta) (V^T - P^T) for tokens 16 hf .. 16 hf + 15; and the two parts of
            // Oq^T summed into the D1 columns (MMA 2 and 3 reuse the other part's columns)
            {
                const uint32_t tok = (C / 2) * hf;
                {
                    float a0[16], a1[16], a2[16], a3[16];
                    tc::ld16(tm + cD1 + C + tok, a0);
                    tc::ld16(tm + cD1 + 3 * C + tok, a1);
                    tc::ld16(tm + cG + C + tok, a2);
                    tc::ld16(tm + cG + 3 * C + tok, a3);
                    tc::wait_ld_regs(a0, a1);
                    tc::wait_ld_regs(a2, a3);
#pragma unroll
                    for (int j = 0; j < C / 2; ++j)
                        a0[j] = __fadd_rn(__fadd_rn(__fadd_rn(a0[j], a1[j]), a2[j]), a3[j]);
                    tc::st16(tm + cD1 + C + tok, a0);
                }
                float pa[16], pb[16], vt[16];
                {
                    float pc[16], pd[16];
                    tc::ld16(tm + cD1 + tok, pa);
                    tc::ld16(tm + cD1 + 2 * C + tok, pb);
                    tc::ld16(tm + cG + tok, pc);
                    tc::ld16(tm + cG + 2 * C + tok, pd);
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) {
                        const int t = (C / 2) * hf + j;
                        vt[j] = t < nt ? load_as_f32<TI>(reinterpret_cast<const TI *>(rawV + t * RP) + v) : 0.0f;
                    }
                    tc::wait_ld_regs(pa, pb);
                    tc::wait_ld_regs(pc, pd);
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) pa[j] = __fadd_rn(__fadd_rn(pa[j], pc[j]), pd[j]);
                }
                if constexpr (GRP) {  // v' = v / c', by one correctly rounded reciprocal of the column's c'
                    const float rc = __frcp_rn(csS[v]);
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) vt[j] = __fmul_rn(vt[j], rc);
                }
#pragma unroll
                for (int j = 0; j < C / 2; ++j) vt[j] = __fmul_rn(betaS[(C / 2) * hf + j], __fsub_rn(vt[j], __fadd_rn(pa[j], pb[j])));
#pragma unroll
                for (int j = 0; j < C / 2; j += 4)
                    put_split4(smem + oA2h, smem + oA2l, tc::kmajor_offset(v, (C / 2) * hf + j, C), vt[j], vt[j + 1],
                               vt[j + 2], vt[j + 3]);
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();  // R^T in place; every copied row of the group has been read (and the decays applied)
            if (!fast && hf == 0) gC[v] = 1.0f;  // nothing pending
            // ---- MMA 2: W^T = R^T [T ; T_lo]^T (thread 0, into the W^T columns) + R_lo^T T^T (thread
            // 32, into the Gram columns), while thread 64 issues the copies of the next group's (or
            // tile's) vectors
            if (tid == 0 || tid == 32) {
                tc::fence_after_sync();
                const bool hi = tid == 0;
                const uint32_t ia = tc::idesc_tf32(128, hi ? 2 * C : C);
                const uint64_t da = hi ? dA2h : dA2l;
                const uint32_t acc = tbase + (hi ? cW : cG);
#pragma unroll
                for (int s = 0; s < C / 8; ++s) tc::mma_tf32(acc, da + 16 * s, dTh + 16 * s, ia, s > 0);
                tc::commit(&bars[1]);
            }
            if (!last) {
                fetch(item, t0 + C, n, 64);
            } else if (nxt < items) {
                fetch(nxt, 0, nxt_n, 64);
            }
            pendm |= 1u << 1;
            if (!wait_bar(1, ph)) {
                failed = true;
                break;
            }
            pendm &= ~(1u << 1);
            tc::fence_after_sync();
            {
                float wa[16], wb[16], wc[16];
                tc::ld16(tm + cW + (C / 2) * hf, wa);
                tc::ld16(tm + cW + C + (C / 2) * hf, wb);
                tc::ld16(tm + cG + (C / 2) * hf, wc);
                tc::wait_ld_regs(wa, wb);
                tc::wait_ld_regs(wc);
#pragma unroll
                for (int j = 0; j < C / 2; ++j) wa[j] = __fadd_rn(__fadd_rn(wa[j], wb[j]), wc[j]);
#pragma unroll
                for (int j = 0; j < C / 2; j += 4)
                    put_split4(smem + oA2h, smem + oA2l, tc::kmajor_offset(v, (C / 2) * hf + j, C), wa[j], wa[j + 1],
                               wa[j + 2], wa[j + 3]);
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            // ---- MMA 3 (thread 0): W^T Bm^T into the W^T columns, now free ([hi*hi + lo*hi |
            // hi*lo]); MMA 4 (thread 32): S^T += W^T Ktil
            if (tid == 0) {
                tc::fence_after_sync();
                const uint32_t i2 = tc::idesc_tf32(128, 2 * C), i1 = tc::idesc_tf32(128, C);
#pragma unroll
                for (int s = 0; s < C / 8; ++s) {
                    tc::mma_tf32(tbase + cW, dA2h + 16 * s, dBh + 16 * s, i2, s > 0);
                    tc::mma_tf32(tbase + cW, dA2l + 16 * s, dBh + 16 * s, i1, true);
                }
                tc::commit(&bars[2]);
            } else if (tid == 32) {
                tc::fence_after_sync();
                const uint32_t idd = tc::idesc_tf32(128, D);
#pragma unroll
                for (int s = 0; s < C / 8; ++s) {
                    const uint64_t ah = dA2h + 16 * s, al = dA2l + 16 * s;
                    const uint64_t kh = dKTh + 16 * s, kl = dKTl + 16 * s;
                    tc::mma_tf32(tbase + cS, ah, kh, idd, true);
                    tc::mma_tf32(tbase + cS, ah, kl, idd, true);
                    tc::mma_tf32(tbase + cS, al, kh, idd, true);
                }
                tc::commit(&bars[6]);
            }
            pendm |= 1u << 2 | 1u << 6;
            if (!wait_bar(2, ph)) {
                failed = true;
                break;
            }
            pendm &= ~(1u << 2);
            tc::fence_after_sync();
            if (o_g) {  // O^T = Oq^T (summed when R was formed) + W^T Bm^T (two parts)
                float oa[16], oc[16], od[16];
                tc::wait_st();  // this thread's Oq^T sums have landed
                tc::ld16(tm + cD1 + C + (C / 2) * hf, oa);
                tc::ld16(tm + cW + (C / 2) * hf, oc);
                tc::ld16(tm + cW + C + (C / 2) * hf, od);
                tc::wait_ld_regs(oa, oc);
                tc::wait_ld_regs(od);
#pragma unroll
                for (int j = 0; j < C / 2; ++j) {
                    oa[j] = __fadd_rn(oa[j], __fadd_rn(oc[j], od[j]));
                    if constexpr (GRP) oa[j] = __fmul_rn(csS[v], oa[j]);  // o = c' o'
                }
                if (M.o_rows && nt == C) {
                    // a full group: rows [t][v] in the T / Bm operand buffers (free until the next
                    // group's operands, which wait until this copy has read them), one tensor copy out
                    TO *ost = reinterpret_cast<TO *>(smem + oTh);
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) store_from_f32<TO>(ost + ((C / 2) * hf + j) * D + v, oa[j]);
                    fence_proxy_async_smem();
                    __syncthreads();
                    if (tid == 0) {
                        tma_store_rows(&M.o, smem + oTh, h, b * L + t0);
                        bulk_store_commit();
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < C / 2; ++j) {
                        const int t = (C / 2) * hf + j;
                        if (t < nt) store_from_f32<TO>(o_g + (((size_t)b * L + t0 + t) * Hv + h) * D + v, oa[j]);
                    }
                }
            }
            if (!wait_bar(6, ph)) {  // MMA 4: the state columns are current
                failed = true;
                break;
            }
            pendm &= ~(1u << 6);
            tc::fence_after_sync();
            ph ^= 1u;
        }
        if (failed) break;
        // ---- the tile's final state (the pending decay applied) to the staging buffers (thread
        // (v, hf): key channels 64 hf .., rows of the pool's layout), then to HBM by bulk copies
        // that run on while the next tile starts (KT and A2 are next written once they are read)
        {
            float *stg = reinterpret_cast<float *>(smem + oKTh);
            int *qflag = reinterpret_cast<int *>(smem + oQflag);
            if (MIX && tid == 0) *qflag = 0;
#pragma unroll
            for (int u0 = 0; u0 < 64; u0 += 32) {
                const int ub = 64 * hf + u0;
                float y[16], y2[16];
                tc::ld16(tm + cS + ub, y);
                tc::ld16(tm + cS + ub + 16, y2);
                tc::wait_ld_regs(y, y2);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    stg[(ub + j) * D + v] = __fmul_rn(y[j], gC[ub + j]);
                    stg[(ub + 16 + j) * D + v] = __fmul_rn(y2[j], gC[ub + 16 + j]);
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if constexpr (!MIX) {
                if (tid == 0) {
                    bulk_s2g(Sg, smem + oKTh, D * D * 4);
                    bulk_store_commit();
                }
            } else {
                // requantise (DAMP Appendix A.4: written once): the absmax of each key channel's row
                // (warp w: rows 16 w .. 16 w + 15, a lane's four columns, then a warp reduction),
                // the scale of its physical row, then thread (v, hf) writes the words of column v
                float *qs = reinterpret_cast<float *>(smem + oQs);
                float *qns = reinterpret_cast<float *>(smem + oQns);
                float *qrc = reinterpret_cast<float *>(smem + oQrc);
                const int lane = tid & 31;
                auto max_nan = [](float a, float b) {
                    float r;
                    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
                    return r;
                };
                float amax = 0.0f;  // lane i: the absmax of row 16 w + i (one scale per row)
                float mg[16];       // DAMP-exact: the lane's maximum of its four columns, row 16 w + i
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int u = 16 * w + i;
                    const float4 x4 = reinterpret_cast<const float4 *>(stg + u * D)[lane];
                    const float m = max_nan(max_nan(fabsf(x4.x), fabsf(x4.y)), max_nan(fabsf(x4.z), fabsf(x4.w)));
                    if constexpr (GRP) {
                        mg[i] = m;
                    } else {
                        const float a = warp_max_abs_nan(m);  // every lane takes part in the reduction
                        amax = lane == i ? a : amax;
                    }
                }
                if constexpr (GRP) {
                    // the maxima over each group's eight lanes (lanes 8 g .. 8 g + 7: columns 32 g ..),
                    // halving the rows at each exchange: at the level of lane bit b the lane keeps the
                    // rows whose bit 3 - b equals its own bit b and sends the others, so that 14
                    // exchanges leave it the group maxima of rows 8 b0 + 4 b1 + 2 b2 + {0, 1}
                    const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
                    float n8[8], n4[4], n2[2];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float keep = b0 ? mg[k + 8] : mg[k], send = b0 ? mg[k] : mg[k + 8];
                        n8[k] = max_nan(keep, __shfl_xor_sync(0xffffffffu, send, 1));
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float keep = b1 ? n8[k + 4] : n8[k], send = b1 ? n8[k] : n8[k + 4];
                        n4[k] = max_nan(keep, __shfl_xor_sync(0xffffffffu, send, 2));
                    }
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float keep = b2 ? n4[k + 2] : n4[k], send = b2 ? n4[k] : n4[k + 2];
                        n2[k] = max_nan(keep, __shfl_xor_sync(0xffffffffu, send, 4));
                    }
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int i = 8 * b0 + 4 * b1 + 2 * b2 + k;
                        const int r = pinv[16 * w + i];
                        if (r >= KHM) qs[(lane >> 3) * D + r] = n2[k];
                    }
                }
                if constexpr (!GRP) {
                    const int r = lane < 16 ? (int)pinv[16 * w + lane] : 0;
                    if (lane < 16 && r >= KHM) qs[r] = amax;
                }
                __syncthreads();
                // the scales of every (group, INT8 row) from the maxima
                constexpr int NGc = GRP ? NGM : 1;
                for (int pq = tid; pq < NGc * (D - KHM); pq += kThreads) {
                    const int g = pq / (D - KHM), r = KHM + pq % (D - KHM);
                    const float a = qs[g * D + r];
                    const uint32_t ab = __float_as_uint(a);
                    const float sv = __fdiv_rn(fmaxf(a, 1e-8f), 127.0f);
                    qs[g * D + r] = sv;
                    qns[g * D + r] = -sv;
                    // fused arithmetic: y = 0 marks a row (group) whose absmax is inf or NaN
                    qrc[g * D + r] = (FUSED && ab >= 0x7f800000u) ? 0.0f : __frcp_rn(sv);
                    if (ab >= 0x7f800000u) *qflag = 1;  // the exact path for the tile
                    reinterpret_cast<float *>(tile_g + 2 * KHM * D + (D - KHM) * D)[GRP ? (r - KHM) * NGM + g : r - KHM] = sv;
                }
                __syncthreads();
                const bool exact = *qflag != 0;
                uint32_t *hw = reinterpret_cast<uint32_t *>(tile_g);
                uint32_t *lw = reinterpret_cast<uint32_t *>(tile_g + 2 * KHM * D);
                const int go = GRP ? (v >> 5) * D : 0;  // column v's scale group
                // thread (v, hf) writes column v of 18 of the 36 word rows (hf = 0: the 8 FP16 pair
                // rows and INT8 quads 0..9; hf = 1: quads 10..27); each batch's loads go ahead of its
                // quantisation and stores
                constexpr int kQuads = (D - KHM) / 4, kQB = 6;
                auto quads = [&](int q0, int q1) {
                    for (int b0 = q0; b0 < q1; b0 += kQB) {
                        float2 x01[kQB], x23[kQB];
                        float4 rc4[kQB], s4[kQB];  // reciprocals; negated scales (IEEE), or scales (exact path)
#pragma unroll
                        for (int i = 0; i < kQB; ++i) {
                            const int qd = min(b0 + i, q1 - 1), r0 = KHM + 4 * qd;
                            const uint32_t pr = pi4[r0 / 4];
                            x01[i] = make_float2(stg[(pr & 0xffu) * D + v], stg[((pr >> 8) & 0xffu) * D + v]);
                            x23[i] = make_float2(stg[((pr >> 16) & 0xffu) * D + v], stg[(pr >> 24) * D + v]);
                            rc4[i] = *reinterpret_cast<const float4 *>(qrc + go + r0);
                            if (exact || !FUSED) s4[i] = *reinterpret_cast<const float4 *>((exact ? qs : qns) + go + r0);
                        }
#pragma unroll
                        for (int i = 0; i < kQB; ++i) {
                            if (b0 + i >= q1) break;
                            uint32_t wd;
                            if (!exact) {
                                if constexpr (FUSED) wd = quant_quad_rcp(x01[i], x23[i], rc4[i]);
                                else wd = quant_quad(x01[i], x23[i], s4[i], rc4[i]);
                            } else {
                                wd = quant_quad_cold<FUSED>(x01[i], x23[i], s4[i], rc4[i]);
                            }
                            lw[(b0 + i) * D + v] = wd;
                        }
                    }
                };
                if (hf == 0) {  // FP16 rows 2 j, 2 j + 1: round to nearest even
                    uint32_t ph[KHM / 4];
#pragma unroll
                    for (int j = 0; j < KHM / 4; ++j) ph[j] = pi4[j];
                    float2 xh[KHM / 2];
#pragma unroll
                    for (int j = 0; j < KHM / 2; ++j) {
                        const uint32_t p2 = ph[j >> 1] >> (16 * (j & 1));
                        xh[j] = make_float2(stg[(p2 & 0xffu) * D + v], stg[((p2 >> 8) & 0xffu) * D + v]);
                    }
#pragma unroll
                    for (int j = 0; j < KHM / 2; ++j) {
                        const __half2 hh = __floats2half2_rn(xh[j].x, xh[j].y);
                        hw[j * D + v] = *reinterpret_cast<const uint32_t *>(&hh);
                    }
                    quads(0, (kQuads - KHM / 2) / 2);
                } else {
                    quads((kQuads - KHM / 2) / 2, kQuads);
                }
            }
        }
    }
    if (failed) {
        // give what is still in flight a bounded time to land before the memory is released
        for (int k = 0; k < kBars; ++k)
            if (pendm >> k & 1u) mbar_wait_bounded(&bars[k], k == 3 ? sph : k == 4 ? iph : k == 5 ? gph : ph);
        if (tid == 0) report_bits(P.status, RS_DEV_PIPE_TIMEOUT);
    }
    if (tid == 0) bulk_store_wait_all();  // the last state copies out have landed
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (w == 0) tc::tmem_dealloc(tbase, kTmemCols);
}

// The driver's tiled tensor-map encoder, reached through the runtime (no link to the driver
// library); null if this driver does not offer it.
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encoder() {
    static const EncodeTiled fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (EncodeTiled) nullptr;
        }
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

// map of a [rows][heads][D] tensor of `esize`-byte elements, box (D + 16 bytes, 1, C)
// (pad: the box is D + 16 bytes wide, the columns past D reading as zeros)
cudaError_t encode_rows(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int heads,
                        int64_t rows, bool pad = true) {
    const EncodeTiled fn = encoder();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)heads * D * esize};
    const cuuint32_t box[3] = {(cuuint32_t)((D * esize + (pad ? 16 : 0)) / esize), 1u, (cuuint32_t)C};
    const cuuint32_t step[3] = {1u, 1u, 1u};
    const CUresult r = fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, step, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename TI>
constexpr CUtensorMapDataType map_type() {
    if constexpr (sizeof(TI) == 4) return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    else if constexpr (std::is_same_v<TI, __half>) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    else return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

template <bool KDA, bool MIX, bool GRP, bool FUSED, typename TI, typename TO, typename PT>
cudaError_t run(PT &P, cudaStream_t s) {
    auto kern = chunk_prefill_kernel<KDA, MIX, GRP, FUSED, TI, TO, PT>;
    const int items = P.B * P.Hv;
    const int64_t rows = (int64_t)P.B * P.L;
    if (items < 1 || rows < 1) return cudaSuccess;
    if (rows > INT32_MAX - C) return cudaErrorNotSupported;  // tensor-copy row coordinates are 32-bit
    ChunkMaps M;
    std::memset(&M, 0, sizeof(M));
    cudaError_t e = encode_rows(&M.k, P.k, map_type<TI>(), (int)sizeof(TI), P.Hk, rows);
    if (e == cudaSuccess) e = encode_rows(&M.q, P.q, map_type<TI>(), (int)sizeof(TI), P.Hk, rows);
    if (e == cudaSuccess) e = encode_rows(&M.v, P.v, map_type<TI>(), (int)sizeof(TI), P.Hv, rows);
    if (e == cudaSuccess && KDA) e = encode_rows(&M.a, P.alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, P.Hv, rows);
    if (e != cudaSuccess) return e;
    if (P.o && (reinterpret_cast<uintptr_t>(P.o) & 15u) == 0 &&
        encode_rows(&M.o, P.o, map_type<TO>(), (int)sizeof(TO), P.Hv, rows, false) == cudaSuccess)
        M.o_rows = 1;  // else each thread stores its outputs
    e = set_dynamic_smem(reinterpret_cast<const void *>(kern), kSmem);
    if (e != cudaSuccess) return e;
    int grid = device_sm_count();
    if (grid > items) grid = items;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmem, s, P, M);
}

}  // namespace

}  // namespace rs
