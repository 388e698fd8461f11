// rs_quant.cuh -- the symmetric INT8 row quantiser shared by the kernels that
// write INT8 codes (DAMP §3.2 Eq. 5-6; dasc Appendix E.1 Eq. 8):
// s = max(a, 1e-8) / 127 with a the row's absmax, code = clip(rne(x / s)).
// The exact quotient and the int8 <-> f32 conversions live in rs_step.cuh;
// this header adds the division-free row scale.
#pragma once

#include "rs_step.cuh"

namespace rs {

// RN(a / 127) for a >= 1e-8 or a = +inf, without a division: q0 = RN(a y)
// with y = RN(1/127), one exact-remainder correction q = RN(q0 + RN(a - q0
// 127) y) (Markstein's correction step).  Checked against the IEEE quotient
// for every finite FP32 a >= 1e-8; +inf is passed through.
__device__ __forceinline__ float div127(float a) {
    constexpr float y = 1.0f / 127.0f;
    const float q0 = __fmul_rn(a, y);
    const float q = __fmaf_rn(__fmaf_rn(-q0, 127.0f, a), y, q0);
    return a == __int_as_float(0x7f800000) ? a : q;
}

// The row scale of the quantiser from the row's absmax a (>= 0 or NaN): a NaN
// absmax takes the 1e-8 floor (fmaxf), an infinite one gives an infinite scale.
__device__ __forceinline__ float row_scale_from_absmax(float a) { return div127(fmaxf(a, 1e-8f)); }

}  // namespace rs
