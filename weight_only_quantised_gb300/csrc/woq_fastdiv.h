// Unsigned 32-bit division by a run-time invariant divisor with one multiply-high, after
// T. Granlund and P. L. Montgomery, "Division by Invariant Integers using
// Multiplication" (PLDI 1994), section 4 (unsigned division, figure 4.1):
//
//   l = ceil(log2 d),  m = floor(2^32 (2^l - d) / d) + 1  (fits 32 bits),
//   t = mulhi(m, n),   n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0)
//
// exact for every 0 <= n < 2^32 and 1 <= d < 2^32.  The host computes (m, l) once per
// launch; the stream-K partition of the GEMV then divides by the CTA count, the block
// count and the group count without the long integer-division sequence.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define WOQ_FD_HD __host__ __device__
#else
#define WOQ_FD_HD
#endif

namespace woq {

struct FastDiv {
  uint32_t d;    // divisor
  uint32_t m;    // multiplier
  uint32_t sh1;  // min(l, 1)
  uint32_t sh2;  // max(l - 1, 0)

  WOQ_FD_HD static FastDiv make(uint32_t divisor) {
    FastDiv f;
    f.d = divisor ? divisor : 1u;
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < (uint64_t)f.d) ++l;  // ceil(log2 d)
    f.m = (uint32_t)((((1ull << l) - f.d) << 32) / f.d + 1);
    f.sh1 = l < 1 ? l : 1u;
    f.sh2 = l > 1 ? l - 1 : 0u;
    return f;
  }

  WOQ_FD_HD uint32_t div(uint32_t n) const {
#if defined(__CUDA_ARCH__)
    const uint32_t t = __umulhi(m, n);
#else
    const uint32_t t = (uint32_t)(((uint64_t)m * n) >> 32);
#endif
    return (t + ((n - t) >> sh1)) >> sh2;
  }
};

}  // namespace woq
