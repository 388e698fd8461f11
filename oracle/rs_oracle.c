/*
 * rs_oracle.c -- plain, slow CPU oracle for the recurrent-state hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (pages, cited by title and section):
 *   [dasc] "dasc: Decay-Aware State Compression for Hybrid Linear-Attention
 *          Serving" (arXiv 2608.30386).
 *   [DAMP] "DAMP: Decay-Aware Mixed-Precision Recurrent-State Quantization"
 *          (arXiv 2608.27513).
 *   [SRA]  "Serving recurrent attention" (Kimi K3 explainer, section 22).
 *
 * Arithmetic: IEEE binary32, round to nearest even, no flush to zero, built
 * with -ffp-contract=off so that every '*' and '+' rounds on its own.  Where a
 * fused multiply-add is meant it is written as fmaf() (correctly rounded by
 * the C library), so the order and the roundings of every result below are
 * fixed by this source alone.
 *
 * Orientation ([DAMP] §3.1): per head the state S has dk rows (key channels)
 * of dv values each, row-major, S[u*dv + v].  One decode step is
 *     S <- diag(a) S;   p = S^T k;   e = v - p;   S <- S + beta k e^T;
 *     o = S^T q  (read from the updated state, [DAMP] §3.1 Eq. 1).
 * Expanding [DAMP] §3.1 Eq. 2, (I - beta k k^T) Lambda S + beta k v^T, gives
 * exactly these lines; [dasc] §3.1 Eq. 1 is the same map on S^T.
 *
 * Reading fixed here (the pages leave the floating-point order open):
 *   - the decay is one multiply per element, S[u][v] * a[u];
 *   - both reductions over u run in ascending u, starting from +0.0f, each
 *     term accumulated with one fused multiply-add, p = fmaf(S[u][v], k[u], p);
 *   - the rank-1 write is S[u][v] = fmaf(beta*k[u], e[v], S[u][v]) with the
 *     product beta*k[u] rounded first.
 *
 * Status bits returned by the batched entry points (same meaning as the
 * device status word of the library, defined independently here):
 *   1 = a slot index out of range (that item is skipped),
 *   2 = an accepted-token count out of range (that item is skipped),
 *   4 = a checkpoint slot out of range (that item is skipped).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define ORC_MAX_D 256

/* ------------------------------------------------------------------------ */
/* One decode step on one state tile (rows in the order given).             */
/* a_stride = 0 gives one decay for the whole head (GDN, [DAMP] §3.1:        */
/* Lambda = alpha I); a_stride = 1 gives one decay per key channel (KDA,     */
/* Lambda = diag(exp g)).  o may be NULL.                                    */
/* ------------------------------------------------------------------------ */
void orc_step_tile_f32(int dk, int dv, float *S, const float *q, const float *k,
                       const float *v, const float *a, int a_stride, float beta,
                       float *o)
{
    float e[ORC_MAX_D];
    int u, c;

    /* S <- diag(a) S */
    for (u = 0; u < dk; ++u) {
        float au = a[(size_t)u * (size_t)a_stride];
        for (c = 0; c < dv; ++c)
            S[(size_t)u * dv + c] = S[(size_t)u * dv + c] * au;
    }
    /* prediction p = S^T k, error e = v - p */
    for (c = 0; c < dv; ++c) {
        float p = 0.0f;
        for (u = 0; u < dk; ++u)
            p = fmaf(S[(size_t)u * dv + c], k[u], p);
        e[c] = v[c] - p;
    }
    /* rank-1 delta-rule write S <- S + beta k e^T */
    for (u = 0; u < dk; ++u) {
        float bk = beta * k[u];
        for (c = 0; c < dv; ++c)
            S[(size_t)u * dv + c] = fmaf(bk, e[c], S[(size_t)u * dv + c]);
    }
    /* readout o = S^T q on the updated state */
    if (o) {
        for (c = 0; c < dv; ++c) {
            float acc = 0.0f;
            for (u = 0; u < dk; ++u)
                acc = fmaf(S[(size_t)u * dv + c], q[u], acc);
            o[c] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Symmetric INT8 row quantiser ([DAMP] §3.2 Eq. 5-6 with b = 8, "x a row of */
/* S"; floor, clip and FP32 arithmetic as in [dasc] Appendix E.1 Eq. 8).     */
/*   a = max_v |x_v|            (a NaN anywhere makes a NaN)                 */
/*   s = max(a, 1e-8) / 127     (fmaxf: a NaN a gives the floor)             */
/*   c_v = clip(round_half_even(x_v / s), -127, 127)                        */
/* Dequantised value: c * s, one FP32 multiply.                              */
/* ------------------------------------------------------------------------ */
static float row_absmax(int n, const float *x)
{
    float a = 0.0f;
    int i;
    for (i = 0; i < n; ++i) {
        float ax = fabsf(x[i]);
        if (isnan(ax) || ax > a)
            a = ax;
    }
    return a;
}

float orc_row_scale(int n, const float *x)
{
    return fmaxf(row_absmax(n, x), 1e-8f) / 127.0f;
}

int8_t orc_quant_code(float x, float s)
{
    float r = rintf(x / s);          /* default rounding: half to even */
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int8_t)r;
}

void orc_quantise_row(int n, const float *x, int8_t *codes, float *scale)
{
    float s = orc_row_scale(n, x);
    int i;
    for (i = 0; i < n; ++i)
        codes[i] = orc_quant_code(x[i], s);
    *scale = s;
}

void orc_dequantise_row(int n, const int8_t *codes, float s, float *x)
{
    int i;
    for (i = 0; i < n; ++i)
        x[i] = (float)codes[i] * s;
}

/* ------------------------------------------------------------------------ */
/* Fused requantisation arithmetic (mode 1) of the mixed layouts.  The pages */
/* fix the quantiser (s = max(a, 1e-8)/127, code = round(x/s) clipped to     */
/* +-127, FP32) and the step (dequantise, decay, update, requantise), not    */
/* how a kernel evaluates x/s or where the decay's rounding falls.  Mode 0   */
/* (above and in the step) takes the IEEE quotient and decays the            */
/* dequantised value.  Mode 1 is the reading a division-free kernel          */
/* implements, with the same scale s:                                        */
/*   - code = the integer nearest to the exact product x * RN(1/s), ties to  */
/*     even (the quotient through the correctly rounded reciprocal, rounded  */
/*     once); rows whose absmax is inf or NaN keep the IEEE quotient;        */
/*   - everything else is mode 0: the step dequantises, x = RN(c * s), and  */
/*     then decays, RN(x * a_u), so the FP32 state before requantisation,    */
/*     its row maxima and scales are those of mode 0 bit for bit.            */
/* A mode-1 code differs from the mode-0 code only where x/s lies within a   */
/* few units of 2^-24 |x/s| of a half-integer (the acceptance allowance is   */
/* 1e-6 max(1, |x/s|)).                                                      */
/* ------------------------------------------------------------------------ */
int8_t orc_quant_code_rcp(float x, float y)
{
    /* a product of two binary32 values is exact in binary64 */
    double r = rint((double)x * (double)y);
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

void orc_quantise_row_m(int n, const float *x, int mode, int8_t *codes, float *scale)
{
    float a = row_absmax(n, x);
    float s = orc_row_scale(n, x);
    int i;
    if (mode == 1 && a <= FLT_MAX) {
        float y = 1.0f / s;
        for (i = 0; i < n; ++i)
            codes[i] = orc_quant_code_rcp(x[i], y);
    } else {
        for (i = 0; i < n; ++i)
            codes[i] = orc_quant_code(x[i], s);
    }
    *scale = s;
}

/* FP16 storage of a high-precision row: round to nearest even, overflow to
 * infinity (IEEE binary16 through the compiler's _Float16). */
static uint16_t f32_to_f16_bits(float x)
{
    _Float16 h = (_Float16)x;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static float f16_bits_to_f32(uint16_t b)
{
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

/* ------------------------------------------------------------------------ */
/* Mixed-precision head tile ([DAMP] §5.2 and Appendix A.4, with one scale   */
/* per INT8 row as in [DAMP] §3.2):                                          */
/*   bytes [0, 2*khi*dv)              : rows 0..khi-1 as FP16                */
/*   bytes [.., + (dk-khi)*dv)        : rows khi..dk-1 as INT8 codes         */
/*   bytes [.., + 4*(dk-khi))         : one FP32 scale per INT8 row          */
/* Rows are physical rows of the permuted state T = P_K S ([DAMP] Appendix   */
/* A.3 Eq. 17, value scaling and value reordering not applied).              */
/* The pages fix that the two regions are contiguous so that they can be     */
/* moved with vector loads and stores ([DAMP] Appendix A.4); the order of    */
/* the values inside a region is left open.  Reading fixed here: rows are    */
/* interleaved by the width of one 32-bit word, so the values of one column  */
/* in 2 consecutive FP16 rows (or 4 consecutive INT8 rows) share a word:     */
/*   FP16 value (r, c), r < khi:  half index ((r/2)*dv + c)*2 + r%2           */
/*   INT8 value (r, c), r >= khi: byte index ((q/4)*dv + c)*4 + q%4, q = r-khi */
/* (khi a multiple of 4).                                                    */
/* ------------------------------------------------------------------------ */
size_t orc_mixed_tile_bytes(int dk, int dv, int khi)
{
    return (size_t)2 * khi * dv + (size_t)(dk - khi) * dv + (size_t)4 * (dk - khi);
}

static size_t hi_offset(int dv, int r, int c)   /* byte offset in the FP16 region */
{
    return (((size_t)(r / 2) * dv + c) * 2 + (size_t)(r % 2)) * 2;
}

static size_t lo_offset(int dv, int q, int c)   /* byte offset in the INT8 region */
{
    return ((size_t)(q / 4) * dv + c) * 4 + (size_t)(q % 4);
}

void orc_mixed_unpack(int dk, int dv, int khi, const uint8_t *tile, float *T)
{
    const uint8_t *hi = tile;
    const uint8_t *lo = tile + (size_t)2 * khi * dv;
    const uint8_t *sc = tile + (size_t)2 * khi * dv + (size_t)(dk - khi) * dv;
    int8_t row[ORC_MAX_D];
    int r, c;
    for (r = 0; r < khi; ++r)
        for (c = 0; c < dv; ++c) {
            uint16_t b;
            memcpy(&b, hi + hi_offset(dv, r, c), 2);
            T[(size_t)r * dv + c] = f16_bits_to_f32(b);
        }
    for (r = khi; r < dk; ++r) {
        float s;
        memcpy(&s, sc + (size_t)(r - khi) * 4, 4);
        for (c = 0; c < dv; ++c)
            row[c] = (int8_t)lo[lo_offset(dv, r - khi, c)];
        orc_dequantise_row(dv, row, s, T + (size_t)r * dv);
    }
}

void orc_mixed_pack_m(int dk, int dv, int khi, int mode, const float *T, uint8_t *tile)
{
    uint8_t *hi = tile;
    uint8_t *lo = tile + (size_t)2 * khi * dv;
    uint8_t *sc = tile + (size_t)2 * khi * dv + (size_t)(dk - khi) * dv;
    int8_t row[ORC_MAX_D];
    int r, c;
    for (r = 0; r < khi; ++r)
        for (c = 0; c < dv; ++c) {
            uint16_t b = f32_to_f16_bits(T[(size_t)r * dv + c]);
            memcpy(hi + hi_offset(dv, r, c), &b, 2);
        }
    for (r = khi; r < dk; ++r) {
        float s;
        orc_quantise_row_m(dv, T + (size_t)r * dv, mode, row, &s);
        for (c = 0; c < dv; ++c)
            lo[lo_offset(dv, r - khi, c)] = (uint8_t)row[c];
        memcpy(sc + (size_t)(r - khi) * 4, &s, 4);
    }
}

void orc_mixed_pack(int dk, int dv, int khi, const float *T, uint8_t *tile)
{
    orc_mixed_pack_m(dk, dv, khi, 0, T, tile);
}

/* Row map of one head ([DAMP] Appendix A.2, Algorithm 1, last step: the
 * selected high-risk key channels are moved to the front; Appendix A.3
 * Eq. 17: the permutation P_K reorders the rows of S).  sel holds the khi
 * selected channels in any order; pi[r] is the logical channel stored in
 * physical row r.  Reading: the pages do not order the channels inside
 * either region; here each region keeps ascending channel order.  Returns -1
 * if sel repeats a channel or names one outside [0, dk). */
int orc_row_map(int dk, int khi, const int16_t *sel, int16_t *pi)
{
    unsigned char chosen[ORC_MAX_D];
    int c, j, r = 0;
    if (dk <= 0 || dk > ORC_MAX_D || khi < 0 || khi > dk) return -1;
    memset(chosen, 0, sizeof chosen);
    for (j = 0; j < khi; ++j) {
        if (sel[j] < 0 || sel[j] >= dk || chosen[sel[j]]) return -1;
        chosen[sel[j]] = 1;
    }
    for (c = 0; c < dk; ++c)        /* the selected region, ascending */
        if (chosen[c]) pi[r++] = (int16_t)c;
    for (c = 0; c < dk; ++c)        /* then the rest, ascending */
        if (!chosen[c]) pi[r++] = (int16_t)c;
    return 0;
}

/* Logical FP32 head S (rows = key channels) <-> mixed tile with row map pi:
 * physical row r holds logical channel pi[r] ([DAMP] Appendix A.2, last step
 * of Algorithm 1; Appendix A.3 Eq. 17). */
int orc_convert_f32_to_mixed_m(int dk, int dv, int khi, int mode, const int16_t *pi,
                               const float *S, uint8_t *tile)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    int r;
    if (!T) return -1;
    for (r = 0; r < dk; ++r)
        memcpy(T + (size_t)r * dv, S + (size_t)pi[r] * dv, (size_t)dv * 4);
    orc_mixed_pack_m(dk, dv, khi, mode, T, tile);
    free(T);
    return 0;
}

int orc_convert_f32_to_mixed(int dk, int dv, int khi, const int16_t *pi,
                             const float *S, uint8_t *tile)
{
    return orc_convert_f32_to_mixed_m(dk, dv, khi, 0, pi, S, tile);
}

int orc_convert_mixed_to_f32(int dk, int dv, int khi, const int16_t *pi,
                             const uint8_t *tile, float *S)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    int r;
    if (!T) return -1;
    orc_mixed_unpack(dk, dv, khi, tile, T);
    for (r = 0; r < dk; ++r)
        memcpy(S + (size_t)pi[r] * dv, T + (size_t)r * dv, (size_t)dv * 4);
    free(T);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Batched decode over a pool.                                               */
/* Pool (one layer): [n_slots][Hv][head_bytes]; item = b*Hv + h, b < B.      */
/* Value head h reads q, k of key head g = h / (Hv/Hk): the Hv/Hk adjacent   */
/* value heads share one key head ([dasc] Appendix B.1).                     */
/* q, k: [B][Hk][dk] f32; v: [B][Hv][dv]; alpha: [B][Hv] (per_channel = 0)   */
/* or [B][Hv][dk] (per_channel = 1); beta: [B][Hv]; o: [B][Hv][dv] or NULL.  */
/* Items [item_begin, item_end) are processed, so callers may split work.   */
/* ------------------------------------------------------------------------ */
static int key_head(int h, int Hk, int Hv) { return h / (Hv / Hk); }

int orc_decode_f32(int B, int Hk, int Hv, int dk, int dv, int per_channel,
                   float *pool, int n_slots, const int32_t *slot_idx,
                   const float *q, const float *k, const float *v,
                   const float *alpha, const float *beta, float *o,
                   int item_begin, int item_end)
{
    int status = 0, it;
    (void)B;
    for (it = item_begin; it < item_end; ++it) {
        int b = it / Hv, h = it % Hv, g = key_head(h, Hk, Hv);
        int32_t slot = slot_idx[b];
        float *S;
        const float *a;
        if (slot < 0 || slot >= n_slots) { status |= 1; continue; }
        S = pool + ((size_t)slot * Hv + h) * (size_t)dk * dv;
        a = per_channel ? alpha + ((size_t)b * Hv + h) * dk : alpha + (size_t)b * Hv + h;
        orc_step_tile_f32(dk, dv, S,
                          q + ((size_t)b * Hk + g) * dk, k + ((size_t)b * Hk + g) * dk,
                          v + ((size_t)b * Hv + h) * dv, a, per_channel ? 1 : 0,
                          beta[(size_t)b * Hv + h],
                          o ? o + ((size_t)b * Hv + h) * dv : NULL);
    }
    return status;
}

/* Mixed-layout decode: dequantise once, one FP32 step in the permuted
 * coordinates of [DAMP] Appendix A.3 Eq. 18 (inputs gathered by pi, the sums
 * over physical rows in ascending row order), requantise once and write back
 * ([DAMP] Appendix A.4 "Fused decoding").  pi: [Hv][dk].  mode: 0 or 1, the
 * requantisation arithmetic (see orc_quant_code_rcp): the modes differ only
 * in how the new codes are rounded. */

int orc_decode_mixed_m(int B, int Hk, int Hv, int dk, int dv, int khi, int per_channel, int mode,
                       uint8_t *pool, int n_slots, const int32_t *slot_idx,
                       const int16_t *pi, const float *q, const float *k, const float *v,
                       const float *alpha, const float *beta, float *o,
                       int item_begin, int item_end)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    float qp[ORC_MAX_D], kp[ORC_MAX_D], ap[ORC_MAX_D];
    size_t tb = orc_mixed_tile_bytes(dk, dv, khi);
    int status = 0, it, r;
    (void)B;
    if (!T) return -1;
    for (it = item_begin; it < item_end; ++it) {
        int b = it / Hv, h = it % Hv, g = key_head(h, Hk, Hv);
        int32_t slot = slot_idx[b];
        const int16_t *ph = pi + (size_t)h * dk;
        const float *qh = q + ((size_t)b * Hk + g) * dk, *kh = k + ((size_t)b * Hk + g) * dk;
        uint8_t *tile;
        if (slot < 0 || slot >= n_slots) { status |= 1; continue; }
        tile = pool + ((size_t)slot * Hv + h) * tb;
        for (r = 0; r < dk; ++r) {
            qp[r] = qh[ph[r]];
            kp[r] = kh[ph[r]];
            ap[r] = per_channel ? alpha[((size_t)b * Hv + h) * dk + ph[r]]
                                : alpha[(size_t)b * Hv + h];
        }
        orc_mixed_unpack(dk, dv, khi, tile, T);
        orc_step_tile_f32(dk, dv, T, qp, kp, v + ((size_t)b * Hv + h) * dv, ap, 1,
                          beta[(size_t)b * Hv + h],
                          o ? o + ((size_t)b * Hv + h) * dv : NULL);
        orc_mixed_pack_m(dk, dv, khi, mode, T, tile);
    }
    free(T);
    return status;
}

int orc_decode_mixed(int B, int Hk, int Hv, int dk, int dv, int khi, int per_channel,
                     uint8_t *pool, int n_slots, const int32_t *slot_idx,
                     const int16_t *pi, const float *q, const float *k, const float *v,
                     const float *alpha, const float *beta, float *o,
                     int item_begin, int item_end)
{
    return orc_decode_mixed_m(B, Hk, Hv, dk, dv, khi, per_channel, 0, pool, n_slots, slot_idx, pi,
                              q, k, v, alpha, beta, o, item_begin, item_end);
}

/* ------------------------------------------------------------------------ */
/* Speculative-token replay ([SRA] "Speculative decoding without state       */
/* snapshots"): the inputs of T_max logged draft tokens are kept; for each   */
/* sequence the first n_accept[b] of them are replayed on the state, which   */
/* is loaded (and dequantised) once and stored (and requantised) once.       */
/* Inputs are [B][T_max][...] versions of the decode inputs; o is            */
/* [B][T_max][Hv][dv] or NULL, rows t >= n_accept[b] are not written.        */
/* ------------------------------------------------------------------------ */
int orc_replay_f32(int B, int T_max, int Hk, int Hv, int dk, int dv, int per_channel,
                   float *pool, int n_slots, const int32_t *slot_idx, const int32_t *n_accept,
                   const float *q, const float *k, const float *v,
                   const float *alpha, const float *beta, float *o,
                   int item_begin, int item_end)
{
    int status = 0, it, t;
    (void)B;
    for (it = item_begin; it < item_end; ++it) {
        int b = it / Hv, h = it % Hv, g = key_head(h, Hk, Hv);
        int32_t slot = slot_idx[b], n = n_accept[b];
        float *S;
        if (slot < 0 || slot >= n_slots) { status |= 1; continue; }
        if (n < 0 || n > T_max) { status |= 2; continue; }
        S = pool + ((size_t)slot * Hv + h) * (size_t)dk * dv;
        for (t = 0; t < n; ++t) {
            size_t bt = (size_t)b * T_max + t;
            const float *a = per_channel ? alpha + (bt * Hv + h) * dk : alpha + bt * Hv + h;
            orc_step_tile_f32(dk, dv, S, q + (bt * Hk + g) * dk, k + (bt * Hk + g) * dk,
                              v + (bt * Hv + h) * dv, a, per_channel ? 1 : 0,
                              beta[bt * Hv + h], o ? o + (bt * Hv + h) * dv : NULL);
        }
    }
    return status;
}

/* mode as in orc_decode_mixed_m (the requantisation arithmetic only). */
int orc_replay_mixed_m(int B, int T_max, int Hk, int Hv, int dk, int dv, int khi, int per_channel,
                       int mode, uint8_t *pool, int n_slots, const int32_t *slot_idx,
                       const int32_t *n_accept, const int16_t *pi, const float *q, const float *k,
                       const float *v, const float *alpha, const float *beta, float *o,
                       int item_begin, int item_end)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    float qp[ORC_MAX_D], kp[ORC_MAX_D], ap[ORC_MAX_D];
    size_t tb = orc_mixed_tile_bytes(dk, dv, khi);
    int status = 0, it, t, r;
    (void)B;
    if (!T) return -1;
    for (it = item_begin; it < item_end; ++it) {
        int b = it / Hv, h = it % Hv, g = key_head(h, Hk, Hv);
        int32_t slot = slot_idx[b], n = n_accept[b];
        const int16_t *ph = pi + (size_t)h * dk;
        uint8_t *tile;
        if (slot < 0 || slot >= n_slots) { status |= 1; continue; }
        if (n < 0 || n > T_max) { status |= 2; continue; }
        if (n == 0) continue;            /* nothing accepted: state untouched */
        tile = pool + ((size_t)slot * Hv + h) * tb;
        for (t = 0; t < n; ++t) {
            size_t bt = (size_t)b * T_max + t;
            const float *qh = q + (bt * Hk + g) * dk, *kh = k + (bt * Hk + g) * dk;
            for (r = 0; r < dk; ++r) {
                qp[r] = qh[ph[r]];
                kp[r] = kh[ph[r]];
                ap[r] = per_channel ? alpha[(bt * Hv + h) * dk + ph[r]] : alpha[bt * Hv + h];
            }
            if (t == 0)
                orc_mixed_unpack(dk, dv, khi, tile, T);
            orc_step_tile_f32(dk, dv, T, qp, kp, v + (bt * Hv + h) * dv, ap, 1,
                              beta[bt * Hv + h], o ? o + (bt * Hv + h) * dv : NULL);
        }
        orc_mixed_pack_m(dk, dv, khi, mode, T, tile);
    }
    free(T);
    return status;
}

int orc_replay_mixed(int B, int T_max, int Hk, int Hv, int dk, int dv, int khi, int per_channel,
                     uint8_t *pool, int n_slots, const int32_t *slot_idx, const int32_t *n_accept,
                     const int16_t *pi, const float *q, const float *k, const float *v,
                     const float *alpha, const float *beta, float *o,
                     int item_begin, int item_end)
{
    return orc_replay_mixed_m(B, T_max, Hk, Hv, dk, dv, khi, per_channel, 0, pool, n_slots, slot_idx,
                              n_accept, pi, q, k, v, alpha, beta, o, item_begin, item_end);
}

/* ------------------------------------------------------------------------ */
/* dasc checkpoints ([dasc] §4.1 and Appendix B "Ragged (Scheme 2)").        */
/* A unit is one head (GDN, unit = 0) or one (head, key channel) row of dv   */
/* values (KDA, unit = 1) of the FP32 state.  keep: [L][n_units] of 0/1.     */
/* r_l = retained units of layer l; offsets o_0 = 0, o_l = o_{l-1} + r_l;    */
/* layer l's units occupy packed positions [o_{l-1}, o_l), in ascending unit */
/* order.  Pool: [L][slots][Hv][dk*dv*4] with layer stride layer_stride      */
/* bytes; checkpoint pool: [ckpt_slots][o_L][unit_bytes].                    */
/* ------------------------------------------------------------------------ */
static size_t unit_bytes_of(int unit, int dk, int dv)
{
    return unit ? (size_t)dv * 4 : (size_t)dk * dv * 4;
}

static int units_per_layer(int unit, int Hv, int dk)
{
    return unit ? Hv * dk : Hv;
}

/* offsets[0..L]: o_0 = 0, o_l = o_{l-1} + r_l */
void orc_plan_offsets(int L, int Hv, int dk, int unit, const uint8_t *keep, int64_t *offsets)
{
    int n = units_per_layer(unit, Hv, dk), l, x;
    offsets[0] = 0;
    for (l = 1; l <= L; ++l) {
        int64_t r = 0;
        for (x = 0; x < n; ++x)
            r += keep[(size_t)(l - 1) * n + x] ? 1 : 0;
        offsets[l] = offsets[l - 1] + r;
    }
}

int orc_ckpt_pack(int L, int Hv, int dk, int dv, int unit, const uint8_t *keep,
                  const uint8_t *pool, int64_t layer_stride, int n_pool_slots,
                  const int32_t *src_slots, const int32_t *dst_ckpt_slots, int n,
                  uint8_t *ckpt, int n_ckpt_slots)
{
    int64_t off[1025];
    int nu = units_per_layer(unit, Hv, dk), i, l, x;
    size_t ub = unit_bytes_of(unit, dk, dv), slot_bytes = (size_t)Hv * dk * dv * 4;
    int status = 0;
    if (L > 1024) return -1;
    orc_plan_offsets(L, Hv, dk, unit, keep, off);
    for (i = 0; i < n; ++i) {
        int32_t s = src_slots[i], d = dst_ckpt_slots[i];
        if (s < 0 || s >= n_pool_slots) { status |= 1; continue; }
        if (d < 0 || d >= n_ckpt_slots) { status |= 4; continue; }
        for (l = 0; l < L; ++l) {
            int64_t j = 0;
            for (x = 0; x < nu; ++x) {
                if (!keep[(size_t)l * nu + x]) continue;
                memcpy(ckpt + ((size_t)d * off[L] + (size_t)(off[l] + j)) * ub,
                       pool + (size_t)l * layer_stride + (size_t)s * slot_bytes + (size_t)x * ub,
                       ub);
                ++j;
            }
        }
    }
    return status;
}

/* dasc-nr restore ([dasc] §4.2): retained units are loaded exactly, omitted
 * units are left at zero (+0.0, all bytes 0x00). */
int orc_ckpt_restore(int L, int Hv, int dk, int dv, int unit, const uint8_t *keep,
                     const uint8_t *ckpt, int n_ckpt_slots, const int32_t *src_ckpt_slots,
                     uint8_t *pool, int64_t layer_stride, int n_pool_slots,
                     const int32_t *dst_slots, int n)
{
    int64_t off[1025];
    int nu = units_per_layer(unit, Hv, dk), i, l, x;
    size_t ub = unit_bytes_of(unit, dk, dv), slot_bytes = (size_t)Hv * dk * dv * 4;
    int status = 0;
    if (L > 1024) return -1;
    orc_plan_offsets(L, Hv, dk, unit, keep, off);
    for (i = 0; i < n; ++i) {
        int32_t s = src_ckpt_slots[i], d = dst_slots[i];
        if (s < 0 || s >= n_ckpt_slots) { status |= 4; continue; }
        if (d < 0 || d >= n_pool_slots) { status |= 1; continue; }
        for (l = 0; l < L; ++l) {
            int64_t j = 0;
            for (x = 0; x < nu; ++x) {
                uint8_t *dst = pool + (size_t)l * layer_stride + (size_t)d * slot_bytes + (size_t)x * ub;
                if (keep[(size_t)l * nu + x]) {
                    memcpy(dst, ckpt + ((size_t)s * off[L] + (size_t)(off[l] + j)) * ub, ub);
                    ++j;
                } else {
                    memset(dst, 0, ub);
                }
            }
        }
    }
    return status;
}

/* ---------------------------------------------------------------------------
 * Checkpoints of whole packed heads ([DAMP] §5.2 layout, [dasc] §4.1 Scheme 2
 * ragged packing): a unit is one head of head_bytes bytes (a mixed tile with
 * its FP16 rows, INT8 codes and scales, copied verbatim).  Same order and
 * offsets as orc_ckpt_pack with head units; restore writes zero bytes to
 * omitted heads, which decode as the zero state.
 * ------------------------------------------------------------------------- */
int orc_ckpt_pack_heads(int L, int Hv, int64_t head_bytes, const uint8_t *keep,
                        const uint8_t *pool, int64_t layer_stride, int n_pool_slots,
                        const int32_t *src_slots, const int32_t *dst_ckpt_slots, int n,
                        uint8_t *ckpt, int n_ckpt_slots)
{
    int64_t off[1025];
    size_t ub = (size_t)head_bytes, slot_bytes = (size_t)Hv * ub;
    int status = 0, i, l, x;
    if (L > 1024) return -1;
    orc_plan_offsets(L, Hv, 1, 0, keep, off);
    for (i = 0; i < n; ++i) {
        int32_t s = src_slots[i], d = dst_ckpt_slots[i];
        if (s < 0 || s >= n_pool_slots) { status |= 1; continue; }
        if (d < 0 || d >= n_ckpt_slots) { status |= 4; continue; }
        for (l = 0; l < L; ++l) {
            int64_t j = 0;
            for (x = 0; x < Hv; ++x) {
                if (!keep[(size_t)l * Hv + x]) continue;
                memcpy(ckpt + ((size_t)d * off[L] + (size_t)(off[l] + j)) * ub,
                       pool + (size_t)l * layer_stride + (size_t)s * slot_bytes + (size_t)x * ub, ub);
                ++j;
            }
        }
    }
    return status;
}

int orc_ckpt_restore_heads(int L, int Hv, int64_t head_bytes, const uint8_t *keep,
                           const uint8_t *ckpt, int n_ckpt_slots, const int32_t *src_ckpt_slots,
                           uint8_t *pool, int64_t layer_stride, int n_pool_slots,
                           const int32_t *dst_slots, int n)
{
    int64_t off[1025];
    size_t ub = (size_t)head_bytes, slot_bytes = (size_t)Hv * ub;
    int status = 0, i, l, x;
    if (L > 1024) return -1;
    orc_plan_offsets(L, Hv, 1, 0, keep, off);
    for (i = 0; i < n; ++i) {
        int32_t s = src_ckpt_slots[i], d = dst_slots[i];
        if (s < 0 || s >= n_ckpt_slots) { status |= 4; continue; }
        if (d < 0 || d >= n_pool_slots) { status |= 1; continue; }
        for (l = 0; l < L; ++l) {
            int64_t j = 0;
            for (x = 0; x < Hv; ++x) {
                uint8_t *dst = pool + (size_t)l * layer_stride + (size_t)d * slot_bytes + (size_t)x * ub;
                if (keep[(size_t)l * Hv + x]) {
                    memcpy(dst, ckpt + ((size_t)s * off[L] + (size_t)(off[l] + j)) * ub, ub);
                    ++j;
                } else {
                    memset(dst, 0, ub);
                }
            }
        }
    }
    return status;
}

/* ---------------------------------------------------------------------------
 * INT8 state checkpoint ([dasc] Appendix E.1, Eq. 8): the retained units of
 * an FP32 state are quantised once at insertion and dequantised once on reuse.
 * One scale per (layer, head, key channel), shared over dv: in this oracle's
 * orientation (rows = key channels) that is one scale per row, the same
 * symmetric quantiser as the mixed layout's INT8 rows (orc_quantise_row).
 *
 * A unit covers R rows of dv values: R = dk for a head (GDN), R = 1 for a
 * key channel (KDA).  Checkpoint slot layout (reading fixed here; the pages
 * give the format, not the byte order):
 *     codes  [o_L][R][dv]  int8, units in packed order (orc_plan_offsets),
 *     scales [o_L][R]      float32,
 * the scales starting right after the codes; a slot occupies
 * orc_ckpt_int8_slot_bytes() bytes (codes + scales, rounded up to 16).
 * Restore: omitted units are +0.0; retained rows are codes[v] * scale.
 * ------------------------------------------------------------------------- */
int64_t orc_ckpt_int8_codes_bytes(int64_t n_kept, int rows, int dv)
{
    return n_kept * rows * dv;
}

int64_t orc_ckpt_int8_slot_bytes(int64_t n_kept, int rows, int dv)
{
    int64_t b = n_kept * rows * ((int64_t)dv + 4);
    return (b + 15) / 16 * 16;
}

int orc_ckpt_pack_int8(int L, int Hv, int dk, int dv, int unit, const uint8_t *keep,
                       const float *pool, int64_t layer_stride_floats, int n_pool_slots,
                       const int32_t *src_slots, const int32_t *dst_ckpt_slots, int n,
                       uint8_t *ckpt, int n_ckpt_slots)
{
    int64_t off[1025];
    int nu = units_per_layer(unit, Hv, dk), R = unit ? 1 : dk, i, l, x, r;
    size_t slot_floats = (size_t)Hv * dk * dv;
    int64_t sb, cb;
    int status = 0;
    if (L > 1024) return -1;
    orc_plan_offsets(L, Hv, dk, unit, keep, off);
    sb = orc_ckpt_int8_slot_bytes(off[L], R, dv);
    cb = orc_ckpt_int8_codes_bytes(off[L], R, dv);
    for (i = 0; i < n; ++i) {
        int32_t s = src_slots[i], d = dst_ckpt_slots[i];
        if (s < 0 || s >= n_pool_slots) { status |= 1; continue; }
        if (d < 0 || d >= n_ckpt_slots) { status |= 4; continue; }
        for (l = 0; l < L; ++l) {
            int64_t j = 0;
            for (x = 0; x < nu; ++x) {
                const float *src;
                if (!keep[(size_t)l * nu + x]) continue;
                /* unit x: head x (R = dk rows) or row x of the slot (R = 1) */
                src = pool + (size_t)l * layer_stride_floats + (size_t)s * slot_floats
                      + (size_t)x * R * dv;
                for (r = 0; r < R; ++r) {
                    int64_t row = (off[l] + j) * R + r;
                    int8_t *codes = (int8_t *)(ckpt + (size_t)d * sb + (size_t)row * dv);
                    float sc;
                    orc_quantise_row(dv, src + (size_t)r * dv, codes, &sc);
                    memcpy(ckpt + (size_t)d * sb + (size_t)cb + (size_t)row * 4, &sc, 4);
                }
                ++j;
            }
        }
    }
    return status;
}

int orc_ckpt_restore_int8(int L, int Hv, int dk, int dv, int unit, const uint8_t *keep,
                          const uint8_t *ckpt, int n_ckpt_slots, const int32_t *src_ckpt_slots,
                          float *pool, int64_t layer_stride_floats, int n_pool_slots,
                          const int32_t *dst_slots, int n)
{
    int64_t off[1025];
    int nu = units_per_layer(unit, Hv, dk), R = unit ? 1 : dk, i, l, x, r;
    size_t slot_floats = (size_t)Hv * dk * dv;
    int64_t sb, cb;
    int status = 0;
    if (L > 1024) return -1;
    orc_plan_offsets(L, Hv, dk, unit, keep, off);
    sb = orc_ckpt_int8_slot_bytes(off[L], R, dv);
    cb = orc_ckpt_int8_codes_bytes(off[L], R, dv);
    for (i = 0; i < n; ++i) {
        int32_t s = src_ckpt_slots[i], d = dst_slots[i];
        if (s < 0 || s >= n_ckpt_slots) { status |= 4; continue; }
        if (d < 0 || d >= n_pool_slots) { status |= 1; continue; }
        for (l = 0; l < L; ++l) {
            int64_t j = 0;
            for (x = 0; x < nu; ++x) {
                float *dst = pool + (size_t)l * layer_stride_floats + (size_t)d * slot_floats
                             + (size_t)x * R * dv;
                if (!keep[(size_t)l * nu + x]) {
                    memset(dst, 0, (size_t)R * dv * 4);
                    continue;
                }
                for (r = 0; r < R; ++r) {
                    int64_t row = (off[l] + j) * R + r;
                    float sc;
                    memcpy(&sc, ckpt + (size_t)s * sb + (size_t)cb + (size_t)row * 4, 4);
                    orc_dequantise_row(dv, (const int8_t *)(ckpt + (size_t)s * sb + (size_t)row * dv),
                                       sc, dst + (size_t)r * dv);
                }
                ++j;
            }
        }
    }
    return status;
}

/* ---------------------------------------------------------------------------
 * DAMP-exact storage ([DAMP] Appendix A.1 "Integer formats" and "Value
 * scaling and reordering", A.3 Eq. 17-18, A.4 "State storage"):
 *   - INT8 rows are quantised in groups of `group` consecutive values along
 *     dv, one FP32 scale per group (the page's group is 32), with the same
 *     symmetric quantiser as above (orc_quantise_row on each group);
 *   - the stored state is T = P_K S D_c^{-1} P_V^T.  The model produces its
 *     value coordinates already in P_V order (A.3: the projections are
 *     rearranged offline), so here the value order is taken as given and
 *     cs[c] = c'_c are the scaling factors in that order (D'_c);
 *   - the step runs on T in the transformed coordinates (Eq. 18): v' =
 *     D'_c^{-1} v (v[c] / cs[c], one IEEE division), the delta-rule update
 *     as in orc_step_tile_f32, and o = D'_c T^T q' (cs[c] * o'[c]).
 * Tile: FP16 and INT8 regions as in the one-scale-per-row tile (same word
 * interleave), then the scales [dk - khi][dv / group] row-major.  With
 * group = dv and cs = 1 this is exactly the one-scale-per-row layout.
 * ------------------------------------------------------------------------- */
size_t orc_damp_tile_bytes(int dk, int dv, int khi, int group)
{
    return (size_t)2 * khi * dv + (size_t)(dk - khi) * dv + (size_t)4 * (dk - khi) * (dv / group);
}

void orc_damp_unpack(int dk, int dv, int khi, int group, const uint8_t *tile, float *T)
{
    const uint8_t *hi = tile;
    const uint8_t *lo = tile + (size_t)2 * khi * dv;
    const uint8_t *sc = tile + (size_t)2 * khi * dv + (size_t)(dk - khi) * dv;
    int ng = dv / group, r, c, gi;
    int8_t row[ORC_MAX_D];
    for (r = 0; r < khi; ++r)
        for (c = 0; c < dv; ++c) {
            uint16_t b;
            memcpy(&b, hi + hi_offset(dv, r, c), 2);
            T[(size_t)r * dv + c] = f16_bits_to_f32(b);
        }
    for (r = khi; r < dk; ++r) {
        for (c = 0; c < dv; ++c)
            row[c] = (int8_t)lo[lo_offset(dv, r - khi, c)];
        for (gi = 0; gi < ng; ++gi) {
            float s;
            memcpy(&s, sc + ((size_t)(r - khi) * ng + gi) * 4, 4);
            orc_dequantise_row(group, row + gi * group, s, T + (size_t)r * dv + gi * group);
        }
    }
}

void orc_damp_pack_m(int dk, int dv, int khi, int group, int mode, const float *T, uint8_t *tile)
{
    uint8_t *hi = tile;
    uint8_t *lo = tile + (size_t)2 * khi * dv;
    uint8_t *sc = tile + (size_t)2 * khi * dv + (size_t)(dk - khi) * dv;
    int ng = dv / group, r, c, gi;
    int8_t row[ORC_MAX_D];
    for (r = 0; r < khi; ++r)
        for (c = 0; c < dv; ++c) {
            uint16_t b = f32_to_f16_bits(T[(size_t)r * dv + c]);
            memcpy(hi + hi_offset(dv, r, c), &b, 2);
        }
    for (r = khi; r < dk; ++r) {
        for (gi = 0; gi < ng; ++gi) {
            float s;
            orc_quantise_row_m(group, T + (size_t)r * dv + gi * group, mode, row + gi * group, &s);
            memcpy(sc + ((size_t)(r - khi) * ng + gi) * 4, &s, 4);
        }
        for (c = 0; c < dv; ++c)
            lo[lo_offset(dv, r - khi, c)] = (uint8_t)row[c];
    }
}

void orc_damp_pack(int dk, int dv, int khi, int group, const float *T, uint8_t *tile)
{
    orc_damp_pack_m(dk, dv, khi, group, 0, T, tile);
}


/* S (logical rows, value order as produced) <-> tile: T[r][c] = S[pi[r]][c]
 * / cs[c] ([DAMP] Appendix A.3 Eq. 17), and back S[pi[r]][c] = T[r][c] * cs[c]. */
int orc_convert_f32_to_damp_m(int dk, int dv, int khi, int group, int mode, const int16_t *pi,
                              const float *cs, const float *S, uint8_t *tile)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    int r, c;
    if (!T) return -1;
    for (r = 0; r < dk; ++r)
        for (c = 0; c < dv; ++c)
            T[(size_t)r * dv + c] = S[(size_t)pi[r] * dv + c] / cs[c];
    orc_damp_pack_m(dk, dv, khi, group, mode, T, tile);
    free(T);
    return 0;
}

int orc_convert_f32_to_damp(int dk, int dv, int khi, int group, const int16_t *pi, const float *cs,
                            const float *S, uint8_t *tile)
{
    return orc_convert_f32_to_damp_m(dk, dv, khi, group, 0, pi, cs, S, tile);
}

int orc_convert_damp_to_f32(int dk, int dv, int khi, int group, const int16_t *pi, const float *cs,
                            const uint8_t *tile, float *S)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    int r, c;
    if (!T) return -1;
    orc_damp_unpack(dk, dv, khi, group, tile, T);
    for (r = 0; r < dk; ++r)
        for (c = 0; c < dv; ++c)
            S[(size_t)pi[r] * dv + c] = T[(size_t)r * dv + c] * cs[c];
    free(T);
    return 0;
}

/* One transformed step on T ([DAMP] Appendix A.3 Eq. 18). */
static void damp_step(int dk, int dv, float *T, const float *qp, const float *kp, const float *v,
                      const float *cs, const float *ap, int a_stride, float beta, float *o)
{
    float vp[ORC_MAX_D], op[ORC_MAX_D];
    int c;
    for (c = 0; c < dv; ++c)
        vp[c] = v[c] / cs[c];
    orc_step_tile_f32(dk, dv, T, qp, kp, vp, ap, a_stride, beta, o ? op : NULL);
    if (o)
        for (c = 0; c < dv; ++c)
            o[c] = cs[c] * op[c];
}

/* Batched decode / replay on DAMP tiles: as orc_decode_mixed_m and
 * orc_replay_mixed_m, with group-wise INT8 scales and value scaling; cs is
 * [Hv][dv] (one vector per head). */
int orc_decode_damp_m(int B, int Hk, int Hv, int dk, int dv, int khi, int group, int per_channel,
                      int mode, uint8_t *pool, int n_slots, const int32_t *slot_idx,
                      const int16_t *pi, const float *cs, const float *q, const float *k,
                      const float *v, const float *alpha, const float *beta, float *o,
                      int item_begin, int item_end)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    float qp[ORC_MAX_D], kp[ORC_MAX_D], ap[ORC_MAX_D];
    size_t tb = orc_damp_tile_bytes(dk, dv, khi, group);
    int status = 0, it, r;
    (void)B;
    if (!T) return -1;
    for (it = item_begin; it < item_end; ++it) {
        int b = it / Hv, h = it % Hv, g = key_head(h, Hk, Hv);
        int32_t slot = slot_idx[b];
        const int16_t *ph = pi + (size_t)h * dk;
        const float *qh = q + ((size_t)b * Hk + g) * dk, *kh = k + ((size_t)b * Hk + g) * dk;
        uint8_t *tile;
        if (slot < 0 || slot >= n_slots) { status |= 1; continue; }
        tile = pool + ((size_t)slot * Hv + h) * tb;
        for (r = 0; r < dk; ++r) {
            qp[r] = qh[ph[r]];
            kp[r] = kh[ph[r]];
            ap[r] = per_channel ? alpha[((size_t)b * Hv + h) * dk + ph[r]] : alpha[(size_t)b * Hv + h];
        }
        orc_damp_unpack(dk, dv, khi, group, tile, T);
        damp_step(dk, dv, T, qp, kp, v + ((size_t)b * Hv + h) * dv, cs + (size_t)h * dv, ap, 1,
                  beta[(size_t)b * Hv + h], o ? o + ((size_t)b * Hv + h) * dv : NULL);
        orc_damp_pack_m(dk, dv, khi, group, mode, T, tile);
    }
    free(T);
    return status;
}

int orc_decode_damp(int B, int Hk, int Hv, int dk, int dv, int khi, int group, int per_channel,
                    uint8_t *pool, int n_slots, const int32_t *slot_idx, const int16_t *pi,
                    const float *cs, const float *q, const float *k, const float *v,
                    const float *alpha, const float *beta, float *o, int item_begin, int item_end)
{
    return orc_decode_damp_m(B, Hk, Hv, dk, dv, khi, group, per_channel, 0, pool, n_slots, slot_idx,
                             pi, cs, q, k, v, alpha, beta, o, item_begin, item_end);
}

int orc_replay_damp_m(int B, int T_max, int Hk, int Hv, int dk, int dv, int khi, int group,
                      int per_channel, int mode, uint8_t *pool, int n_slots, const int32_t *slot_idx,
                      const int32_t *n_accept, const int16_t *pi, const float *cs, const float *q,
                      const float *k, const float *v, const float *alpha, const float *beta, float *o,
                      int item_begin, int item_end)
{
    float *T = (float *)malloc((size_t)dk * dv * 4);
    float qp[ORC_MAX_D], kp[ORC_MAX_D], ap[ORC_MAX_D];
    size_t tb = orc_damp_tile_bytes(dk, dv, khi, group);
    int status = 0, it, t, r;
    (void)B;
    if (!T) return -1;
    for (it = item_begin; it < item_end; ++it) {
        int b = it / Hv, h = it % Hv, g = key_head(h, Hk, Hv);
        int32_t slot = slot_idx[b], n = n_accept[b];
        const int16_t *ph = pi + (size_t)h * dk;
        uint8_t *tile;
        if (slot < 0 || slot >= n_slots) { status |= 1; continue; }
        if (n < 0 || n > T_max) { status |= 2; continue; }
        if (n == 0) continue;
        tile = pool + ((size_t)slot * Hv + h) * tb;
        for (t = 0; t < n; ++t) {
            size_t bt = (size_t)b * T_max + t;
            const float *qh = q + (bt * Hk + g) * dk, *kh = k + (bt * Hk + g) * dk;
            for (r = 0; r < dk; ++r) {
                qp[r] = qh[ph[r]];
                kp[r] = kh[ph[r]];
                ap[r] = per_channel ? alpha[(bt * Hv + h) * dk + ph[r]] : alpha[bt * Hv + h];
            }
            if (t == 0)
                orc_damp_unpack(dk, dv, khi, group, tile, T);
            damp_step(dk, dv, T, qp, kp, v + (bt * Hv + h) * dv, cs + (size_t)h * dv, ap, 1,
                      beta[bt * Hv + h], o ? o + (bt * Hv + h) * dv : NULL);
        }
        orc_damp_pack_m(dk, dv, khi, group, mode, T, tile);
    }
    free(T);
    return status;
}

int orc_replay_damp(int B, int T_max, int Hk, int Hv, int dk, int dv, int khi, int group,
                    int per_channel, uint8_t *pool, int n_slots, const int32_t *slot_idx,
                    const int32_t *n_accept, const int16_t *pi, const float *cs, const float *q,
                    const float *k, const float *v, const float *alpha, const float *beta, float *o,
                    int item_begin, int item_end)
{
    return orc_replay_damp_m(B, T_max, Hk, Hv, dk, dv, khi, group, per_channel, 0, pool, n_slots,
                             slot_idx, n_accept, pi, cs, q, k, v, alpha, beta, o, item_begin, item_end);
}
