// rs_plans.cu -- host-side selection-plan builders of the C ABI.
//
// dasc ("dasc: Decay-Aware State Compression for Hybrid Linear-Attention
// Serving"): static log-decays and retention horizons from the gate weights
// (§3.3 Eq. 2-3), the retention mask H_s > W_max (§4.1) and the suffix-refresh
// window (§4.2 Eq. 7).  DAMP ("DAMP: Decay-Aware Mixed-Precision
// Recurrent-State Quantization"): the local quantisation error of each key
// channel (§5.1 Eq. 14, with the storage quantiser: one INT8 scale per row),
// the accumulated-error risk under the observed decays (§5.1 Eq. 15), and the
// budgeted top-K_hi selection of FP16 channels per head.
//
// Plans are built once, offline, on the host; arithmetic is fp64 from FP32
// inputs, except the quantiser, which is the FP32 storage quantiser itself.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <numeric>
#include <vector>

#include "../../include/recurrent_state.h"

namespace {

double softplus(double x) { return x < 30.0 ? std::log1p(std::exp(x)) : x + std::log1p(std::exp(-x)); }

double static_log_decay(int gate, double A_log, double d, double a_s) {
    if (gate == RS_GATE_STD) return -std::exp(A_log) * softplus(a_s + d);
    return -5.0 / (1.0 + std::exp(-std::exp(A_log) * (a_s + d)));  // l * sigmoid(...), l = -5
}

// Storage quantiser of one row (FP32): s = max(absmax, 1e-8) / 127,
// code = clip(rne(x / s), -127, 127); returns sum over the row of
// (code * s - x)^2 in fp64.
double row_error(const float *x, int n) {
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        const float ax = std::fabs(x[i]);
        if (std::isnan(ax) || ax > a) a = ax;
    }
    const float s = std::fmax(a, 1e-8f) / 127.0f;
    double e = 0.0;
    for (int i = 0; i < n; ++i) {
        float r = std::nearbyint(x[i] / s);
        r = std::fmin(std::fmax(r, -127.0f), 127.0f);
        const double diff = (double)(r * s) - (double)x[i];
        e += diff * diff;
    }
    return e;
}

}  // namespace

extern "C" {

rs_status rs_dasc_horizons(int32_t gate, const float *A_log, const float *d_bias, int64_t n_units,
                           double a_s, double epsilon, double *H) {
    if ((gate != RS_GATE_STD && gate != RS_GATE_K3) || n_units < 0 || !(epsilon > 0.0 && epsilon < 1.0))
        return RS_ERR_INVALID_ARG;
    if (n_units > 0 && (!A_log || !d_bias || !H)) return RS_ERR_INVALID_ARG;
    const double le = std::log(epsilon);
    for (int64_t u = 0; u < n_units; ++u) H[u] = le / static_log_decay(gate, A_log[u], d_bias[u], a_s);
    return RS_OK;
}

rs_status rs_dasc_keep(const double *H, int64_t n_units, double W_max, uint8_t *keep) {
    if (n_units < 0 || (n_units > 0 && (!H || !keep))) return RS_ERR_INVALID_ARG;
    for (int64_t u = 0; u < n_units; ++u) keep[u] = H[u] > W_max ? 1 : 0;
    return RS_OK;
}

rs_status rs_dasc_refresh_window(const double *H, const uint8_t *keep, int64_t n_units, int64_t W_max,
                                 int64_t n_prefix, int64_t *W_replay) {
    if (n_units < 0 || W_max < 4 || n_prefix < 0 || !W_replay || (n_units > 0 && (!H || !keep)))
        return RS_ERR_INVALID_ARG;
    int64_t widest = 0;
    bool any = false;
    for (int64_t u = 0; u < n_units; ++u) {
        if (keep[u]) continue;
        any = true;
        const double h = H[u];
        int64_t w;
        if (std::isnan(h)) return RS_ERR_INVALID_ARG;
        if (h >= (double)W_max) {
            w = W_max;  // next_pow2(h) >= h >= W_max: clamped
        } else if (h <= 0.0) {
            w = 4;  // next_pow2 maps zero to 4; clamped up to 4
        } else {
            int64_t p = 1;
            while ((double)p < h) p *= 2;
            w = std::min<int64_t>(std::max<int64_t>(p, 4), W_max);
        }
        widest = std::max(widest, w);
    }
    *W_replay = any ? std::min(n_prefix, widest) : 0;
    return RS_OK;
}

rs_status rs_damp_risk_scores(const float *states, const float *decays, int32_t n_anchors, int32_t dk,
                              int32_t dv, int32_t horizon, double *C) {
    if (n_anchors <= 0 || dk <= 0 || dv <= 0 || horizon < 0 || !states || !C || (horizon > 0 && !decays))
        return RS_ERR_INVALID_ARG;
    std::fill(C, C + dk, 0.0);
    for (int32_t n = 0; n < n_anchors; ++n) {
        const float *S = states + (size_t)n * dk * dv;
        const float *a = decays + (size_t)n * horizon * dk;
        for (int32_t u = 0; u < dk; ++u) {
            double w = 1.0, prod = 1.0;
            for (int32_t j = 0; j < horizon; ++j) {
                const double ar = a[(size_t)j * dk + u];
                prod *= ar * ar;
                w += prod;
            }
            C[u] += row_error(S + (size_t)u * dv, dv) * w;
        }
    }
    for (int32_t u = 0; u < dk; ++u) C[u] /= n_anchors;
    return RS_OK;
}

rs_status rs_damp_select_hi_rows(const double *C, int32_t n_heads, int32_t dk, int32_t k_hi, int16_t *hi_rows) {
    if (n_heads < 0 || dk <= 0 || k_hi < 0 || k_hi > dk || dk > 32767 ||
        (n_heads > 0 && (!C || (k_hi > 0 && !hi_rows))))
        return RS_ERR_INVALID_ARG;
    std::vector<int32_t> idx((size_t)dk);
    for (int32_t h = 0; h < n_heads; ++h) {
        const double *c = C + (size_t)h * dk;
        for (int32_t u = 0; u < dk; ++u)
            if (std::isnan(c[u])) return RS_ERR_INVALID_ARG;
        std::iota(idx.begin(), idx.end(), 0);
        std::stable_sort(idx.begin(), idx.end(), [&](int32_t x, int32_t y) { return c[x] > c[y]; });
        std::sort(idx.begin(), idx.begin() + k_hi);
        for (int32_t i = 0; i < k_hi; ++i) hi_rows[(size_t)h * k_hi + i] = (int16_t)idx[i];
    }
    return RS_OK;
}

}  // extern "C"
