// rs_api.cu -- host side of the C ABI declared in include/recurrent_state.h:
// layout and plan objects, argument validation, status codes, and dispatch to
// the kernel launchers.  No exception crosses the ABI; every entry point
// returns an rs_status.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/recurrent_state.h"
#include "rs_internal.h"
#include "rs_ckpt_int8.h"
#include "rs_damp.h"

struct rs_layout {
    rs_layout_params p;
    std::vector<int16_t> pi;  // [Hv][dk], physical row -> key channel
    size_t head_bytes;
    int32_t group = 0;        // DAMP-exact layout: values per INT8 scale group (0: one scale per row)
    std::vector<float> cs;    // DAMP-exact layout: value-scaling factors [Hv][dv]
    int32_t quant = RS_QUANT_IEEE;  // requantisation arithmetic of a mixed layout
};


namespace {

thread_local std::string g_last_cuda_error;

rs_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
    return RS_ERR_CUDA;
}

rs_status launch_fail(cudaError_t e) {
    if (e == cudaErrorNotSupported) return RS_ERR_UNSUPPORTED;
    return cuda_fail(e);
}

}  // namespace

namespace rs {
int32_t fail_cuda(cudaError_t e) { return cuda_fail(e); }
int32_t fail_launch(cudaError_t e) { return launch_fail(e); }
}  // namespace rs

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t mixed_head_bytes(int dk, int dv, int khi) {
    return (size_t)2 * khi * dv + (size_t)(dk - khi) * dv + (size_t)4 * (dk - khi);
}

int dtype_size(int32_t dt) {
    switch (dt) {
        case RS_F32: return 4;
        case RS_BF16: return 2;
        case RS_F16: return 2;
        default: return 0;
    }
}

struct DevAttr {
    int sms = 0, smem = 0;
};
std::mutex g_attr_mu;
DevAttr g_attr[64];

DevAttr &attr_for_current() {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_attr_mu);
    DevAttr &a = g_attr[dev & 63];
    if (a.sms == 0) {
        cudaDeviceGetAttribute(&a.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&a.smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return a;
}

}  // namespace

namespace rs {
int device_sm_count() { return attr_for_current().sms; }
int device_max_smem_optin() { return attr_for_current().smem; }

cudaError_t set_dynamic_smem(const void *fn, int bytes) {
    struct Entry {
        const void *fn;
        int dev, bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (Entry &x : done)
        if (x.fn == fn && x.dev == dev) {
            if (x.bytes >= bytes) return cudaSuccess;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e == cudaSuccess) x.bytes = bytes;
            return e;
        }
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.push_back({fn, dev, bytes});
    return e;
}
}  // namespace rs

extern "C" {

const char *rs_status_string(rs_status s) {
    switch (s) {
        case RS_OK: return "ok";
        case RS_ERR_INVALID_ARG: return "invalid argument";
        case RS_ERR_UNSUPPORTED: return "unsupported combination";
        case RS_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case RS_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

const char *rs_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

const char *rs_version(void) { return "0.1.0"; }

// ---------------------------------------------------------------------------
// layouts
// ---------------------------------------------------------------------------
rs_status rs_layout_create(rs_layout **out, const rs_layout_params *p, const int16_t *hi_rows) {
    if (!out || !p) return RS_ERR_INVALID_ARG;
    *out = nullptr;
    if (p->kind != RS_LAYOUT_FP32 && p->kind != RS_LAYOUT_MIXED_FP16_INT8) return RS_ERR_INVALID_ARG;
    if (p->dk <= 0 || p->dv <= 0 || p->num_v_heads <= 0 || p->num_qk_heads <= 0) return RS_ERR_INVALID_ARG;
    if (p->num_v_heads % p->num_qk_heads != 0) return RS_ERR_INVALID_ARG;
    if (p->dk > 256 || p->dv > 256) return RS_ERR_INVALID_ARG;
    if (p->dk != p->dv) return RS_ERR_UNSUPPORTED;
    if (p->dk != 64 && p->dk != 128) return RS_ERR_UNSUPPORTED;
    const int Hv = p->num_v_heads, dk = p->dk;
    rs_layout *l = new (std::nothrow) rs_layout;
    if (!l) return RS_ERR_INVALID_ARG;
    l->p = *p;
    l->pi.resize((size_t)Hv * dk);
    if (p->kind == RS_LAYOUT_FP32) {
        if (p->k_hi != 0) { delete l; return RS_ERR_INVALID_ARG; }
        for (int h = 0; h < Hv; ++h)
            for (int r = 0; r < dk; ++r) l->pi[(size_t)h * dk + r] = (int16_t)r;
        l->head_bytes = (size_t)4 * dk * p->dv;
    } else {
        if (p->k_hi < 0 || p->k_hi > dk || (p->k_hi % 4) != 0 || !hi_rows) { delete l; return RS_ERR_INVALID_ARG; }
        if ((size_t)Hv * dk > (size_t)rs::kMaxRowMap) { delete l; return RS_ERR_UNSUPPORTED; }
        std::vector<uint8_t> seen(dk);
        for (int h = 0; h < Hv; ++h) {
            std::fill(seen.begin(), seen.end(), 0);
            for (int j = 0; j < p->k_hi; ++j) {
                const int c = hi_rows[(size_t)h * p->k_hi + j];
                if (c < 0 || c >= dk || seen[c]) { delete l; return RS_ERR_INVALID_ARG; }
                seen[c] = 1;
            }
            // selected channels first, then the rest, each ascending
            int r = 0;
            for (int c = 0; c < dk; ++c)
                if (seen[c]) l->pi[(size_t)h * dk + r++] = (int16_t)c;
            for (int c = 0; c < dk; ++c)
                if (!seen[c]) l->pi[(size_t)h * dk + r++] = (int16_t)c;
        }
        l->head_bytes = mixed_head_bytes(dk, p->dv, p->k_hi);
    }
    *out = l;
    return RS_OK;
}

rs_status rs_layout_create_damp(rs_layout **out, const rs_layout_params *p, const int16_t *hi_rows,
                                int32_t group, const float *value_scales) {
    if (!out || !p) return RS_ERR_INVALID_ARG;
    *out = nullptr;
    if (p->kind != RS_LAYOUT_MIXED_FP16_INT8 || group <= 0 || p->dv % group != 0) return RS_ERR_INVALID_ARG;
    if (group != rs::kDampGroup) return RS_ERR_UNSUPPORTED;
    if ((size_t)p->num_v_heads * p->dv > (size_t)rs::kMaxValueScales) return RS_ERR_UNSUPPORTED;
    const size_t ncs = (size_t)p->num_v_heads * (size_t)(p->dv > 0 ? p->dv : 0);
    if (value_scales)
        for (size_t i = 0; i < ncs; ++i)
            if (!(value_scales[i] > 0.0f) || !std::isfinite(value_scales[i])) return RS_ERR_INVALID_ARG;
    rs_layout *l = nullptr;
    const rs_status st = rs_layout_create(&l, p, hi_rows);
    if (st != RS_OK) return st;
    l->group = group;
    l->cs.assign(ncs, 1.0f);
    if (value_scales) std::copy(value_scales, value_scales + ncs, l->cs.begin());
    l->head_bytes = (size_t)2 * p->k_hi * p->dv + (size_t)(p->dk - p->k_hi) * p->dv +
                    (size_t)4 * (p->dk - p->k_hi) * (p->dv / group);
    *out = l;
    return RS_OK;
}

rs_status rs_layout_set_quant(rs_layout *l, int32_t mode) {
    if (!l || (mode != RS_QUANT_IEEE && mode != RS_QUANT_FUSED)) return RS_ERR_INVALID_ARG;
    if (l->p.kind == RS_LAYOUT_FP32 && mode != RS_QUANT_IEEE) return RS_ERR_INVALID_ARG;
    l->quant = mode;
    return RS_OK;
}

rs_status rs_layout_quant(const rs_layout *l, int32_t *mode) {
    if (!l || !mode) return RS_ERR_INVALID_ARG;
    *mode = l->quant;
    return RS_OK;
}

rs_status rs_layout_destroy(rs_layout *l) {
    delete l;
    return RS_OK;
}

rs_status rs_layout_head_bytes(const rs_layout *l, size_t *bytes) {
    if (!l || !bytes) return RS_ERR_INVALID_ARG;
    *bytes = l->head_bytes;
    return RS_OK;
}

rs_status rs_layout_row_map(const rs_layout *l, int16_t *pi) {
    if (!l || !pi) return RS_ERR_INVALID_ARG;
    std::memcpy(pi, l->pi.data(), l->pi.size() * sizeof(int16_t));
    return RS_OK;
}

rs_status rs_layout_bits_per_value(const rs_layout *l, double *bits) {
    if (!l || !bits) return RS_ERR_INVALID_ARG;
    *bits = 8.0 * (double)l->head_bytes / ((double)l->p.dk * (double)l->p.dv);
    return RS_OK;
}

// ---------------------------------------------------------------------------
// decode / replay
// ---------------------------------------------------------------------------
static rs_status prefill_common(const rs_layout *l, int32_t per_channel_decay, void *pool, int64_t n_slots,
                                const int32_t *slot_idx, int32_t B, int32_t L, const int32_t *n_tokens,
                                const void *q, const void *k, const void *v, int32_t in_dtype,
                                const float *alpha, const float *beta, void *o, int32_t out_dtype,
                                int32_t *status, void *stream, bool chunked);

static rs_status step_common(const rs_layout *l, bool kda, bool replay, void *pool, int64_t n_slots,
                             const int32_t *slot_idx, int32_t B, int32_t T_max,
                             const int32_t *n_accept, const void *q, const void *k, const void *v,
                             int32_t in_dtype, const float *alpha, const float *beta, void *o,
                             int32_t out_dtype, int32_t *status, void *stream) {
    if (!l) return RS_ERR_INVALID_ARG;
    if (B < 0 || n_slots < 0 || n_slots > INT32_MAX) return RS_ERR_INVALID_ARG;
    if (T_max < 1 || T_max > rs::kMaxTokens) return RS_ERR_INVALID_ARG;
    if (dtype_size(in_dtype) == 0 || (out_dtype != RS_F32 && out_dtype != RS_BF16))
        return RS_ERR_INVALID_ARG;
    const int Hv = l->p.num_v_heads, Hk = l->p.num_qk_heads, D = l->p.dk;
    if ((int64_t)B * Hv > INT32_MAX / 2) return RS_ERR_INVALID_ARG;
    if (B == 0) return RS_OK;
    if (!pool || !slot_idx || !q || !k || !v || !alpha || !beta) return RS_ERR_INVALID_ARG;
    if (replay && !n_accept) return RS_ERR_INVALID_ARG;
    // bulk-copy sources must be 16-byte aligned
    if (!aligned16(pool) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return RS_ERR_MISALIGNED;
    if (kda && !aligned16(alpha)) return RS_ERR_MISALIGNED;
    if ((D * dtype_size(in_dtype)) % 16 != 0) return RS_ERR_UNSUPPORTED;

    rs::StepLaunch L;
    L.D = D;
    L.khi = l->p.kind == RS_LAYOUT_FP32 ? -1 : l->p.k_hi;
    L.kda = kda;
    L.in_dt = in_dtype;
    L.out_dt = out_dtype;
    L.fused = l->p.kind != RS_LAYOUT_FP32 && l->quant == RS_QUANT_FUSED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    auto fill = [&](rs::StepParams &P) {
        P.pool = pool;
        P.n_slots = n_slots;
        P.slot_idx = slot_idx;
        P.n_accept = n_accept;
        P.q = q;
        P.k = k;
        P.v = v;
        P.alpha = alpha;
        P.beta = beta;
        P.o = o;
        P.status = status;
        P.B = B;
        P.Hk = Hk;
        P.Hv = Hv;
        P.T_max = T_max;
        P.replay = replay ? 1 : 0;
        P.header_bytes = 0;
        P.region_bytes = 0;
        P.stages = 0;
    };
    cudaError_t e;
    if (l->p.kind == RS_LAYOUT_FP32) {
        rs::StepParams P;
        fill(P);
        e = D == 128 ? rs::launch_step_f32_d128(L, P, s) : rs::launch_step_f32_d64(L, P, s);
    } else {
        if (l->group) {  // DAMP-exact layout
            // a multi-token replay is a prefill chunk of T_max tokens with
            // n_accept[b] of them applied (same arithmetic, same status bits)
            if (replay)
                return prefill_common(l, kda ? 1 : 0, pool, n_slots, slot_idx, B, T_max, n_accept, q, k, v,
                                      in_dtype, alpha, beta, o, out_dtype, status, stream, false);
            static thread_local rs::StepParamsDamp P;
            fill(P);
            for (size_t i = 0; i < l->pi.size(); ++i) P.pi[i] = (uint8_t)l->pi[i];
            std::copy(l->cs.begin(), l->cs.end(), P.cs);
            e = rs::launch_step_damp_decode(L, P, s);
        } else {
            static thread_local rs::StepParamsPi P;
            fill(P);
            for (size_t i = 0; i < l->pi.size(); ++i) P.pi[i] = (uint8_t)l->pi[i];
            e = (replay || T_max > 1) ? rs::launch_step_mixed_replay(L, P, s)
                                      : rs::launch_step_mixed_decode(L, P, s);
        }
    }
    if (e != cudaSuccess) return launch_fail(e);
    return RS_OK;
}

rs_status rs_gdn_decode_update(const rs_layout *l, void *pool, int64_t n_slots, const int32_t *slot_idx,
                               int32_t B, const void *q, const void *k, const void *v,
                               int32_t in_dtype, const float *alpha, const float *beta, void *o,
                               int32_t out_dtype, int32_t *status, void *stream) {
    return step_common(l, false, false, pool, n_slots, slot_idx, B, 1, nullptr, q, k, v, in_dtype,
                       alpha, beta, o, out_dtype, status, stream);
}

rs_status rs_kda_decode_update(const rs_layout *l, void *pool, int64_t n_slots, const int32_t *slot_idx,
                               int32_t B, const void *q, const void *k, const void *v,
                               int32_t in_dtype, const float *alpha, const float *beta, void *o,
                               int32_t out_dtype, int32_t *status, void *stream) {
    return step_common(l, true, false, pool, n_slots, slot_idx, B, 1, nullptr, q, k, v, in_dtype,
                       alpha, beta, o, out_dtype, status, stream);
}

rs_status rs_spec_replay_update(const rs_layout *l, int32_t per_channel_decay, void *pool,
                                int64_t n_slots, const int32_t *slot_idx, int32_t B, int32_t T_max,
                                const int32_t *n_accept, const void *q, const void *k, const void *v,
                                int32_t in_dtype, const float *alpha, const float *beta, void *o,
                                int32_t out_dtype, int32_t *status, void *stream) {
    if (per_channel_decay != 0 && per_channel_decay != 1) return RS_ERR_INVALID_ARG;
    return step_common(l, per_channel_decay == 1, true, pool, n_slots, slot_idx, B, T_max, n_accept,
                       q, k, v, in_dtype, alpha, beta, o, out_dtype, status, stream);
}

rs_status rs_prefill_update(const rs_layout *l, int32_t per_channel_decay, void *pool, int64_t n_slots,
                            const int32_t *slot_idx, int32_t B, int32_t L, const int32_t *n_tokens,
                            const void *q, const void *k, const void *v, int32_t in_dtype,
                            const float *alpha, const float *beta, void *o, int32_t out_dtype,
                            int32_t *status, void *stream) {
    return prefill_common(l, per_channel_decay, pool, n_slots, slot_idx, B, L, n_tokens, q, k, v, in_dtype,
                          alpha, beta, o, out_dtype, status, stream, false);
}

rs_status rs_prefill_chunked_update(const rs_layout *l, int32_t per_channel_decay, void *pool,
                                    int64_t n_slots, const int32_t *slot_idx, int32_t B, int32_t L,
                                    const int32_t *n_tokens, const void *q, const void *k, const void *v,
                                    int32_t in_dtype, const float *alpha, const float *beta, void *o,
                                    int32_t out_dtype, int32_t *status, void *stream) {
    return prefill_common(l, per_channel_decay, pool, n_slots, slot_idx, B, L, n_tokens, q, k, v, in_dtype,
                          alpha, beta, o, out_dtype, status, stream, true);
}

static rs_status prefill_common(const rs_layout *l, int32_t per_channel_decay, void *pool, int64_t n_slots,
                                const int32_t *slot_idx, int32_t B, int32_t L, const int32_t *n_tokens,
                                const void *q, const void *k, const void *v, int32_t in_dtype,
                                const float *alpha, const float *beta, void *o, int32_t out_dtype,
                                int32_t *status, void *stream, bool chunked) {
    if (!l || (per_channel_decay != 0 && per_channel_decay != 1)) return RS_ERR_INVALID_ARG;
    if (B < 0 || L < 0 || n_slots < 0 || n_slots > INT32_MAX) return RS_ERR_INVALID_ARG;
    if (dtype_size(in_dtype) == 0 || (out_dtype != RS_F32 && out_dtype != RS_BF16)) return RS_ERR_INVALID_ARG;
    const int Hv = l->p.num_v_heads, Hk = l->p.num_qk_heads, D = l->p.dk;
    if ((int64_t)B * Hv > INT32_MAX / 2) return RS_ERR_INVALID_ARG;
    if (B == 0 || L == 0) return RS_OK;
    if (!pool || !slot_idx || !q || !k || !v || !alpha || !beta) return RS_ERR_INVALID_ARG;
    if (!aligned16(pool) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(alpha))
        return RS_ERR_MISALIGNED;
    rs::StepLaunch Ln;
    Ln.D = D;
    Ln.khi = l->p.kind == RS_LAYOUT_FP32 ? -1 : l->p.k_hi;
    Ln.kda = per_channel_decay == 1;
    Ln.in_dt = in_dtype;
    Ln.out_dt = out_dtype;
    Ln.fused = l->p.kind != RS_LAYOUT_FP32 && l->quant == RS_QUANT_FUSED;
    auto fill = [&](rs::PrefillParams &P) {
        P.pool = pool;
        P.n_slots = n_slots;
        P.slot_idx = slot_idx;
        P.n_tokens = n_tokens;
        P.q = q;
        P.k = k;
        P.v = v;
        P.alpha = alpha;
        P.beta = beta;
        P.o = o;
        P.status = status;
        P.B = B;
        P.Hk = Hk;
        P.Hv = Hv;
        P.L = L;
        for (size_t i = 0; i < l->pi.size() && i < (size_t)rs::kMaxRowMap; ++i) P.pi[i] = (uint8_t)l->pi[i];
    };
    cudaError_t e;
    if (chunked) {  // the tensor-core form: FP32 layout, or the mixed ones with 16 FP16 rows
        if (D != 128 || (l->p.kind != RS_LAYOUT_FP32 && l->p.k_hi != 16)) return RS_ERR_UNSUPPORTED;
        if (l->group) {  // DAMP-exact: groups of 32 and value scaling
            if (l->group != rs::kDampGroup) return RS_ERR_UNSUPPORTED;
            static thread_local rs::PrefillParamsDamp P;
            fill(P);
            std::copy(l->cs.begin(), l->cs.end(), P.cs);
            e = rs::launch_prefill_chunked_damp(Ln, P, static_cast<cudaStream_t>(stream));
        } else {
            static thread_local rs::PrefillParams P;
            fill(P);
            e = rs::launch_prefill_chunked(Ln, P, static_cast<cudaStream_t>(stream));
        }
    } else if (l->group) {  // DAMP-exact layout: group scales and value-scaling factors
        static thread_local rs::PrefillParamsDamp P;
        fill(P);
        std::copy(l->cs.begin(), l->cs.end(), P.cs);
        e = rs::launch_prefill_damp(Ln, P, static_cast<cudaStream_t>(stream));
    } else {
        static thread_local rs::PrefillParams P;
        fill(P);
        e = rs::launch_prefill(Ln, P, static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return launch_fail(e);
    return RS_OK;
}

// ---------------------------------------------------------------------------
// conversion
// ---------------------------------------------------------------------------
rs_status rs_state_convert(const rs_layout *src_l, const void *src_pool, const rs_layout *dst_l,
                           void *dst_pool, int64_t n_slots, const int32_t *slots, int32_t n,
                           int32_t *status, void *stream) {
    if (!src_l || !dst_l || n < 0 || n_slots < 0 || n_slots > INT32_MAX) return RS_ERR_INVALID_ARG;
    const rs_layout_params &a = src_l->p, &b = dst_l->p;
    if (a.dk != b.dk || a.dv != b.dv || a.num_v_heads != b.num_v_heads) return RS_ERR_INVALID_ARG;
    if (n == 0) return RS_OK;
    if (!src_pool || !dst_pool || !slots) return RS_ERR_INVALID_ARG;
    if (!aligned16(src_pool) || !aligned16(dst_pool)) return RS_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (a.kind == b.kind) {
        if (a.kind == RS_LAYOUT_MIXED_FP16_INT8 &&
            (a.k_hi != b.k_hi || src_l->pi != dst_l->pi || src_l->group != dst_l->group || src_l->cs != dst_l->cs))
            return RS_ERR_UNSUPPORTED;
        e = rs::launch_copy_heads(src_pool, dst_pool, (int64_t)src_l->head_bytes, slots, n, n_slots,
                                  a.num_v_heads, status, s);
    } else {
        const rs_layout *mixed = a.kind == RS_LAYOUT_MIXED_FP16_INT8 ? src_l : dst_l;
        if (mixed->group) {  // DAMP-exact layout
            static thread_local rs::ConvertParamsDamp P;
            P.src = src_pool;
            P.dst = dst_pool;
            P.n_slots = n_slots;
            P.slots = slots;
            P.status = status;
            P.n = n;
            P.Hv = a.num_v_heads;
            P.to_mixed = b.kind == RS_LAYOUT_MIXED_FP16_INT8 ? 1 : 0;
            P.fused = mixed->quant == RS_QUANT_FUSED ? 1 : 0;
            for (size_t i = 0; i < mixed->pi.size(); ++i) P.pi[i] = (uint8_t)mixed->pi[i];
            std::copy(mixed->cs.begin(), mixed->cs.end(), P.cs);
            e = rs::launch_convert_damp(a.dk, mixed->p.k_hi, P, s);
            if (e != cudaSuccess) return launch_fail(e);
            return RS_OK;
        }
        static thread_local rs::ConvertParamsPi P;
        P.src = src_pool;
        P.dst = dst_pool;
        P.n_slots = n_slots;
        P.slots = slots;
        P.status = status;
        P.n = n;
        P.Hv = a.num_v_heads;
        P.to_mixed = b.kind == RS_LAYOUT_MIXED_FP16_INT8 ? 1 : 0;
        P.fused = mixed->quant == RS_QUANT_FUSED ? 1 : 0;
        for (size_t i = 0; i < mixed->pi.size(); ++i) P.pi[i] = (uint8_t)mixed->pi[i];
        e = rs::launch_convert(a.dk, mixed->p.k_hi, P, s);
    }
    if (e != cudaSuccess) return launch_fail(e);
    return RS_OK;
}

// ---------------------------------------------------------------------------
// checkpoint plans
// ---------------------------------------------------------------------------
rs_status rs_plan_create(rs_plan **out, const rs_layout *l, int32_t num_layers, int32_t unit,
                         const uint8_t *keep) {
    if (!out || !l || !keep || num_layers <= 0 || num_layers >= 2048) return RS_ERR_INVALID_ARG;
    *out = nullptr;
    if (unit != RS_UNIT_HEAD && unit != RS_UNIT_CHANNEL) return RS_ERR_INVALID_ARG;
    if (l->p.kind != RS_LAYOUT_FP32 && unit != RS_UNIT_HEAD) return RS_ERR_UNSUPPORTED;
    rs_plan *p = new (std::nothrow) rs_plan;
    if (!p) return RS_ERR_INVALID_ARG;
    p->L = num_layers;
    p->unit = unit;
    p->Hv = l->p.num_v_heads;
    p->dk = l->p.dk;
    p->dv = l->p.dv;
    p->head_bytes = l->head_bytes;
    p->nu = unit == RS_UNIT_HEAD ? p->Hv : p->Hv * p->dk;
    p->unit_bytes = unit == RS_UNIT_HEAD ? (int64_t)l->head_bytes : (int64_t)p->dv * 4;
    if (p->nu >= (1 << 20)) { delete p; return RS_ERR_UNSUPPORTED; }
    p->offsets.assign((size_t)num_layers + 1, 0);
    p->all_pidx.assign((size_t)num_layers * p->nu, -1);
    for (int lyr = 0; lyr < num_layers; ++lyr) {
        int64_t r = 0;
        for (int x = 0; x < p->nu; ++x) {
            const uint8_t kbit = keep[(size_t)lyr * p->nu + x];
            if (kbit > 1) { delete p; return RS_ERR_INVALID_ARG; }
            if (kbit) {
                p->all_pidx[(size_t)lyr * p->nu + x] = (int32_t)(p->offsets[lyr] + r);
                p->kept_unit.push_back((int32_t)((lyr << 20) | x));
                ++r;
            }
        }
        p->offsets[lyr + 1] = p->offsets[lyr] + r;
    }
    // Page-locked copy of the table for rs_ckpt_pack_noalloc, whose copy into
    // its fixed device array must not stage through pageable memory (such a
    // copy can synchronise with the stream).  Best effort: without a CUDA
    // device (or for a plan beyond that call's limit) none is made, and that
    // call then returns RS_ERR_UNSUPPORTED.
    const size_t nk = p->kept_unit.size();
    if (nk > 0 && (int64_t)nk <= rs::kNoallocTableEntries) {
        void *h = nullptr;
        if (cudaHostAlloc(&h, nk * sizeof(int32_t), cudaHostAllocPortable) == cudaSuccess) {
            std::memcpy(h, p->kept_unit.data(), nk * sizeof(int32_t));
            p->h_kept_pinned = static_cast<int32_t *>(h);
        } else {
            cudaGetLastError();  // leave no error behind for the caller's next CUDA call
        }
    }
    *out = p;
    return RS_OK;
}

rs_status rs_plan_destroy(rs_plan *p) {
    if (!p) return RS_OK;
    if (p->d_kept) cudaFree(p->d_kept);
    if (p->d_all) cudaFree(p->d_all);
    if (p->h_kept_pinned) cudaFreeHost(p->h_kept_pinned);
    delete p;
    return RS_OK;
}

rs_status rs_plan_offsets(const rs_plan *p, int64_t *offsets, int64_t *unit_bytes) {
    if (!p) return RS_ERR_INVALID_ARG;
    if (offsets) std::memcpy(offsets, p->offsets.data(), p->offsets.size() * sizeof(int64_t));
    if (unit_bytes) *unit_bytes = p->unit_bytes;
    return RS_OK;
}

rs_status rs_plan_upload(rs_plan *p) {
    if (!p) return RS_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (p->device == dev) return RS_OK;
    if (p->device >= 0) return RS_ERR_UNSUPPORTED;  // uploaded to another device already
    const size_t nk = std::max<size_t>(p->kept_unit.size(), 1), na = p->all_pidx.size();
    if ((e = cudaMalloc(&p->d_kept, nk * sizeof(int32_t))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMalloc(&p->d_all, na * sizeof(int32_t))) != cudaSuccess) {
        cudaFree(p->d_kept);
        p->d_kept = nullptr;
        return cuda_fail(e);
    }
    if (!p->kept_unit.empty() &&
        (e = cudaMemcpy(p->d_kept, p->kept_unit.data(), p->kept_unit.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaMemcpy(p->d_all, p->all_pidx.data(), na * sizeof(int32_t), cudaMemcpyHostToDevice)) !=
        cudaSuccess)
        return cuda_fail(e);
    p->device = dev;
    return RS_OK;
}

static rs_status ckpt_common(const rs_plan *p, bool pack, const void *src, void *dst,
                             int64_t layer_stride_bytes, int64_t n_pool_slots, int64_t n_ckpt_slots,
                             const int32_t *pool_slots, const int32_t *ckpt_slots, int32_t n,
                             int32_t *status, void *stream) {
    if (!p || n < 0 || n_pool_slots < 0 || n_ckpt_slots < 0) return RS_ERR_INVALID_ARG;
    if (n == 0) return RS_OK;
    // A plan that retains nothing has empty checkpoint slots: the checkpoint
    // pointer is never dereferenced and may be NULL.
    const bool empty_ckpt = p->offsets.back() == 0;
    const void *ckpt_ptr = pack ? static_cast<const void *>(dst) : src;
    const void *pool_ptr = pack ? src : static_cast<const void *>(dst);
    if (!pool_ptr || !pool_slots || !ckpt_slots || (!ckpt_ptr && !empty_ckpt)) return RS_ERR_INVALID_ARG;
    if (!aligned16(pool_ptr) || !aligned16(ckpt_ptr) || (layer_stride_bytes & 15)) return RS_ERR_MISALIGNED;
    const int64_t slot_bytes = (int64_t)p->Hv * (int64_t)p->head_bytes;
    if (p->L > 1 && layer_stride_bytes < slot_bytes * n_pool_slots) return RS_ERR_INVALID_ARG;
    int dev = 0;
    cudaGetDevice(&dev);
    if (p->device != dev) return RS_ERR_INVALID_ARG;  // rs_plan_upload first
    rs::CkptParams P;
    P.src = static_cast<const uint8_t *>(src);
    P.dst = static_cast<uint8_t *>(dst);
    P.layer_stride = layer_stride_bytes;
    P.slot_bytes = slot_bytes;
    P.unit_bytes = p->unit_bytes;
    P.ckpt_slot_bytes = p->offsets.back() * p->unit_bytes;
    P.n_pool_slots = n_pool_slots;
    P.n_ckpt_slots = n_ckpt_slots;
    P.n_kept = p->offsets.back();
    P.n_all = (int64_t)p->L * p->nu;
    P.kept_unit = p->d_kept;
    P.all_pidx = p->d_all;
    P.pool_slots = pool_slots;
    P.ckpt_slots = ckpt_slots;
    P.status = status;
    P.n = n;
    P.units_per_layer = p->nu;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = pack ? rs::launch_ckpt_pack(P, s) : rs::launch_ckpt_restore(P, s);
    if (e != cudaSuccess) return launch_fail(e);
    return RS_OK;
}

rs_status rs_ckpt_pack(const rs_plan *p, const void *pool, int64_t layer_stride_bytes,
                       int64_t n_pool_slots, const int32_t *src_slots, const int32_t *dst_ckpt_slots,
                       int32_t n, void *ckpt_pool, int64_t n_ckpt_slots, int32_t *status,
                       void *stream) {
    return ckpt_common(p, true, pool, ckpt_pool, layer_stride_bytes, n_pool_slots, n_ckpt_slots,
                       src_slots, dst_ckpt_slots, n, status, stream);
}

rs_status rs_ckpt_restore(const rs_plan *p, const void *ckpt_pool, int64_t n_ckpt_slots,
                          const int32_t *src_ckpt_slots, void *pool, int64_t layer_stride_bytes,
                          int64_t n_pool_slots, const int32_t *dst_slots, int32_t n, int32_t *status,
                          void *stream) {
    return ckpt_common(p, false, ckpt_pool, pool, layer_stride_bytes, n_pool_slots, n_ckpt_slots,
                       dst_slots, src_ckpt_slots, n, status, stream);
}

static int64_t int8_rows_per_unit(const rs_plan *p) { return p->unit == RS_UNIT_HEAD ? p->dk : 1; }
// A plan on the FP32 layout: its heads are dk x dv floats (a mixed head is smaller).
static bool plan_fp32(const rs_plan *p) { return p->head_bytes == (size_t)p->dk * p->dv * 4; }

rs_status rs_ckpt_int8_bytes(const rs_plan *p, int64_t *codes_bytes, int64_t *slot_bytes) {
    if (!p) return RS_ERR_INVALID_ARG;
    if (!plan_fp32(p)) return RS_ERR_UNSUPPORTED;
    const int64_t rows = p->offsets.back() * int8_rows_per_unit(p);
    if (codes_bytes) *codes_bytes = rows * p->dv;
    if (slot_bytes) *slot_bytes = (rows * (p->dv + 4) + 15) / 16 * 16;
    return RS_OK;
}

static rs_status ckpt_int8_common(const rs_plan *p, bool pack, const void *src, void *dst,
                                  int64_t layer_stride_bytes, int64_t n_pool_slots, int64_t n_ckpt_slots,
                                  const int32_t *pool_slots, const int32_t *ckpt_slots, int32_t n,
                                  int32_t *status, void *stream) {
    if (!p || n < 0 || n_pool_slots < 0 || n_ckpt_slots < 0) return RS_ERR_INVALID_ARG;
    if (!plan_fp32(p) || (p->dv != 64 && p->dv != 128)) return RS_ERR_UNSUPPORTED;
    if (n == 0) return RS_OK;
    const bool empty_ckpt = p->offsets.back() == 0;
    const void *ckpt_ptr = pack ? static_cast<const void *>(dst) : src;
    const void *pool_ptr = pack ? src : static_cast<const void *>(dst);
    if (!pool_ptr || !pool_slots || !ckpt_slots || (!ckpt_ptr && !empty_ckpt)) return RS_ERR_INVALID_ARG;
    if (!aligned16(pool_ptr) || !aligned16(ckpt_ptr) || (layer_stride_bytes & 15)) return RS_ERR_MISALIGNED;
    const int64_t slot_bytes = (int64_t)p->Hv * (int64_t)p->head_bytes;
    if (p->L > 1 && layer_stride_bytes < slot_bytes * n_pool_slots) return RS_ERR_INVALID_ARG;
    int dev = 0;
    cudaGetDevice(&dev);
    if (p->device != dev) return RS_ERR_INVALID_ARG;  // rs_plan_upload first
    int64_t codes = 0, sb = 0;
    rs_ckpt_int8_bytes(p, &codes, &sb);
    int rows_log2 = 0;
    while ((int64_t(1) << rows_log2) < int8_rows_per_unit(p)) ++rows_log2;
    if ((int64_t(1) << rows_log2) != int8_rows_per_unit(p)) return RS_ERR_UNSUPPORTED;
    rs::Int8CkptParams P;
    P.src = static_cast<const uint8_t *>(src);
    P.dst = static_cast<uint8_t *>(dst);
    P.layer_stride = layer_stride_bytes;
    P.slot_bytes = slot_bytes;
    P.unit_bytes = p->unit_bytes;
    P.ckpt_slot_bytes = sb;
    P.codes_bytes = codes;
    P.n_pool_slots = n_pool_slots;
    P.n_ckpt_slots = n_ckpt_slots;
    P.n_kept = p->offsets.back();
    P.n_all = (int64_t)p->L * p->nu;
    P.kept_unit = p->d_kept;
    P.all_pidx = p->d_all;
    P.pool_slots = pool_slots;
    P.ckpt_slots = ckpt_slots;
    P.status = status;
    P.n = n;
    P.units_per_layer = p->nu;
    P.rows_log2 = rows_log2;
    P.dv = p->dv;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = pack ? rs::launch_ckpt_pack_int8(P, s) : rs::launch_ckpt_restore_int8(P, s);
    if (e != cudaSuccess) return launch_fail(e);
    return RS_OK;
}

rs_status rs_ckpt_pack_int8(const rs_plan *p, const void *pool, int64_t layer_stride_bytes,
                            int64_t n_pool_slots, const int32_t *src_slots, const int32_t *dst_ckpt_slots,
                            int32_t n, void *ckpt_pool, int64_t n_ckpt_slots, int32_t *status,
                            void *stream) {
    return ckpt_int8_common(p, true, pool, ckpt_pool, layer_stride_bytes, n_pool_slots, n_ckpt_slots,
                            src_slots, dst_ckpt_slots, n, status, stream);
}

rs_status rs_ckpt_restore_int8(const rs_plan *p, const void *ckpt_pool, int64_t n_ckpt_slots,
                               const int32_t *src_ckpt_slots, void *pool, int64_t layer_stride_bytes,
                               int64_t n_pool_slots, const int32_t *dst_slots, int32_t n,
                               int32_t *status, void *stream) {
    return ckpt_int8_common(p, false, ckpt_pool, pool, layer_stride_bytes, n_pool_slots, n_ckpt_slots,
                            dst_slots, src_ckpt_slots, n, status, stream);
}

}  // extern "C"
