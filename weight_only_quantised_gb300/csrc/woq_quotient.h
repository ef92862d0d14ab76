// The activation quantiser's quotient without a division.
//
// The code of a value x in a row with scale s = RN(amax / 127) is rne(RN(x / s)): round half
// to even of the IEEE fp32 quotient.  The kernels have rc = RN(1 / s) and form
//     t = RN(x rc),   r = RN(x - t s) (one fused multiply-add),   u = RN(t + r rc) (another),
// the correction step of the division by Newton iteration with a fused multiply-add that
// P. Markstein describes ("Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990; "IA-64 and Elementary Functions", 2000).
// rne(u) is then the code: for every bf16 amax >= 2^-116 and every bf16 x with |x| <= amax,
// rne(u) equals rne(RN(x / s)) (tests/quotient_check.cpp enumerates all of them; below
// 2^-116 the residual can fall into fp32's subnormal range and two codes differ).  The
// kernels evaluate these three operations in pairs (fp32x2); this scalar form is the
// definition the host test checks.
#pragma once

#include <math.h>

#if defined(__CUDACC__)
#define WOQ_QUOT_HD __host__ __device__
#else
#define WOQ_QUOT_HD
#endif

namespace woq {

// Smallest row maximum for which rne(corrected_quotient) is the quantiser's code.
constexpr float kQuotientMinAmax = 0x1p-116f;

WOQ_QUOT_HD inline float corrected_quotient(float x, float s, float rc) {
  const float t = x * rc;
  const float r = fmaf(-t, s, x);
  return fmaf(r, rc, t);
}

}  // namespace woq
