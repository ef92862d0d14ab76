// Checks woq::FastDiv (division by an invariant divisor with one multiply-high) against
// the plain unsigned division: edge divisors and numerators, random pairs, and all small
// pairs.  Built and run by tests/test_fastdiv.py with the host compiler.
#include "woq_fastdiv.h"
#include <cstdio>
#include <cstdint>
#include <initializer_list>
int main() {
  uint64_t s = 88172645463325252ull; auto rnd = [&]() { s ^= s << 13; s ^= s >> 7; s ^= s << 17; return (uint32_t)s; };
  uint32_t ds[] = {1u, 2u, 3u, 5u, 7u, 40u, 128u, 136u, 152u, 304u, 641u, 47520u, 65535u, 65536u, 65537u, 0x7fffffffu, 0x80000000u, 0x80000001u, 0xfffffffeu, 0xffffffffu};
  long bad = 0, n_checks = 0;
  auto check = [&](uint32_t d, uint32_t n) { woq::FastDiv f = woq::FastDiv::make(d); ++n_checks; if (f.div(n) != n / d) { if (bad < 5) printf("d %u n %u: %u != %u\n", d, n, f.div(n), n / d); ++bad; } };
  for (uint32_t d : ds) { for (uint32_t n : {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 2 * d, 0xfffffffeu, 0xffffffffu}) check(d, n); for (int i = 0; i < 20000; ++i) check(d, rnd()); }
  for (int j = 0; j < 20000; ++j) { uint32_t d = rnd() >> (rnd() % 32); if (!d) d = 1; for (int i = 0; i < 50; ++i) check(d, rnd()); uint32_t k = rnd() % 1000; check(d, d * k); check(d, d * k - 1); }
  for (uint32_t d = 1; d < 2000; ++d) for (uint32_t n = 0; n < 5000; n += 7) check(d, n);
  printf("%ld checks, %ld bad\n", n_checks, bad);
  return bad != 0;
}
