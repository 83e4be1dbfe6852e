// E4M3 quantisation helpers shared by the row quantiser and the GEMM epilogue
// that writes the E4M3 combine payload: the scale of a row (or block) and the
// correctly rounded division by it.
#pragma once

#include <cuda_runtime.h>

namespace moe {

// scale = amax / 448 (the largest finite E4M3 value), 1 for an all-zero row.
__device__ __forceinline__ float row_scale(float amax) { return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f; }

// Row divisor: x / s correctly rounded (round to nearest even), as the
// quantisation rule defines it.  For s >= 2^-96 the quotient comes from the
// reciprocal r = RN(1/s) and one correction with the exact FMA residual:
// q0 = RN(x r), e = x - q0 s (exact), q = RN(q0 + e r).  By Markstein's
// theorem (a quotient within one ulp, corrected once with a reciprocal within
// half an ulp, is the correctly rounded quotient, barring underflow and
// overflow) this is RN(x / s); here |x| <= 448 s, so nothing overflows, and an
// underflowing quotient is far below 2^-10, where every E4M3 code is a zero.
// Smaller scales divide with __fdiv_rn.
struct RowDiv {
    float s, r;
    bool fast;
};

__device__ __forceinline__ RowDiv row_div(float s) {
    RowDiv d;
    d.s = s;
    d.r = __frcp_rn(s);
    d.fast = s >= 0x1p-96f;
    return d;
}

template <bool FAST>
__device__ __forceinline__ float div_rn(const RowDiv& d, float x) {
    if (!FAST) return __fdiv_rn(x, d.s);
    const float q0 = x * d.r;
    const float e = fmaf(-q0, d.s, x);
    return fmaf(e, d.r, q0);
}

}  // namespace moe
