// Checks the quantiser's division-free quotient (woq_quotient.h) against the definition: for
// every bf16 amax in [2^-116, 2^121) (all 128 significands, every exponent), s = RN(amax / 127)
// and rc = RN(1 / s), and every bf16 x with |x| <= amax (both signs), rne of the corrected
// quotient equals rne of the IEEE quotient x / s.  It also counts the values where the
// uncorrected t = RN(x rc) would round to another code, and shows that below 2^-116 the
// correction can fail.  Built and run by tests/test_quotient.py (no FP contraction).
#include "woq_quotient.h"
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>

static float bf16(uint32_t b) { float f; std::memcpy(&f, &b, 4); return f; }

static long sweep(int e_lo, int e_hi, long* checks, long* t_wrong) {
  long bad = 0;
  for (int e = e_lo; e <= e_hi; ++e) {
    for (uint32_t f = 0; f < 128; ++f) {
      const float amax = std::ldexp(1.0f + f / 128.0f, e);
      const float s = amax / 127.0f;
      const float rc = 1.0f / s;
      for (uint32_t b = 1; b < 0x7F80u; ++b) {
        const float xa = bf16(b << 16);
        if (xa > amax) break;
        for (int sg = 0; sg < 2; ++sg) {
          const float x = sg ? -xa : xa;
          const float want = std::nearbyint(x / s);  // round half to even, the default mode
          ++*checks;
          if (std::nearbyint(woq::corrected_quotient(x, s, rc)) != want) ++bad;
          if (std::nearbyint(x * rc) != want) ++*t_wrong;
        }
      }
    }
  }
  return bad;
}

int main() {
  long checks = 0, t_wrong = 0, c2 = 0, t2 = 0;
  const long bad = sweep(-116, 120, &checks, &t_wrong);
  const long bad_low = sweep(-119, -117, &c2, &t2);
  printf("%ld checks, %ld where rne(x rc) differs, %ld bad; below 2^-116: %ld bad of %ld\n", checks, t_wrong, bad,
         bad_low, c2);
  return bad != 0;
}
