// Arithmetic shared by the quantize-prepass kernels.
#pragma once
#include <cuda_runtime.h>

namespace ditattn {

// Scales for which div_by_scale below gives the codes exactly: for every quotient that can change
// a code (|x / s| >= 2^-12) the reciprocal, the product and the remainder (a multiple of about
// 2^(e(s) + e(q) - 47), so at least 2^-147 here) are representable without underflow. Outside
// this range the kernels divide with __fdiv_rn.
__device__ __forceinline__ bool scale_in_fast_range(float s) { return s >= 0x1p-88f && s <= 0x1p+120f; }

// x / s rounded to nearest even, given r = RN(1/s) (the correctly rounded reciprocal). Markstein's
// division theorem (P. Markstein, IBM J. Res. Dev. 34(1), 1990; the division-with-FMA theorem in
// Muller et al., "Handbook of Floating-Point Arithmetic"): if q is within one ulp of x / s, the
// remainder is exact as one FMA and RN(q + remainder * r) = RN(x / s). The first guess RN(x * r)
// can be up to two ulps away, so one correction brings it within one ulp and a second one, where
// the theorem applies, rounds it correctly. It holds when no value underflows. The quantizers only
// need the value for |x / s| >= 2^-12: smaller quotients encode to a zero code (INT8 rounds below
// 0.5 to 0, E4M3 rounds below 2^-10 to a signed zero), and for those only the sign matters.
// The remainder is formed as q * s - x and added times -r: the same values as x - q * s times r
// (round to nearest is symmetric), but for x = -0 the exact zero remainder (+0) times -r is -0, so
// the quotient keeps x's sign of zero as IEEE division does (x - q * s would give +0 + -0 = +0 and
// an E4M3 code 0x00 instead of 0x80). A nonzero x keeps its sign in every step.
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float q1 = __fmaf_rn(__fmaf_rn(q0, s, -x), -r, q0);
  return __fmaf_rn(__fmaf_rn(q1, s, -x), -r, q1);
}

// div_by_scale on two values at once, with the packed float32 pairs of the FMA pipes: each lane
// takes the same IEEE steps (round-to-nearest products and fused multiply-adds, subnormals kept),
// so each result equals div_by_scale's, sign of zero included (the packed FMA takes no negated
// operands, so -x costs one packed multiply). ZERO_SIGN = false drops that multiply and forms the
// remainder as x - q * s, which gives +0 for x = -0: only for INT8 codes, which have one zero.
template <bool ZERO_SIGN = true>
__device__ __forceinline__ float2 div2_by_scale(float2 x, float2 s, float2 r) {
  const float2 q0 = __fmul2_rn(x, r);
  if constexpr (ZERO_SIGN) {
    const float2 nx = __fmul2_rn(x, make_float2(-1.0f, -1.0f)), nr = make_float2(-r.x, -r.y);
    const float2 q1 = __ffma2_rn(__ffma2_rn(q0, s, nx), nr, q0);
    return __ffma2_rn(__ffma2_rn(q1, s, nx), nr, q1);
  } else {
    const float2 ns = make_float2(-s.x, -s.y);
    const float2 q1 = __ffma2_rn(__ffma2_rn(q0, ns, x), r, q0);
    return __ffma2_rn(__ffma2_rn(q1, ns, x), r, q1);
  }
}

// amax / qmax rounded to nearest even, for the block scales (qmax 127 or 448): div_by_scale with the
// correctly rounded reciprocal of the constant, for amax in [2^-100, 2^120], where the products and
// remainders neither underflow nor overflow; IEEE division outside that range (and for 0).
__device__ __forceinline__ float scale_of(float amax, float qmax, float rcp_qmax) {
  if (amax >= 0x1p-100f && amax <= 0x1p+120f) return div_by_scale(amax, qmax, rcp_qmax);
  return __fdiv_rn(amax, qmax);
}

}  // namespace ditattn
