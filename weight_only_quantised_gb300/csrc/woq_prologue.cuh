// Prologue fusions of the activation quantisation ("Doubling LLM token rates in
// ComfyUI", section "Optimizing the Linear Kernel": the RMSNorm or SwiGLU before a
// linear is folded into its input quantisation, so the tensor between them never goes
// to memory).  Both produce bf16 h, which is then quantised exactly like a
// bf16 activation.  Every step is an IEEE fp32 operation (or integer arithmetic), so
// the result is fixed bit for bit:
//
//   RMSNorm: a bf16 x is a 2^c with a an integer below 256, so x^2 = a^2 2^(2c) exactly;
//     per row, C = the largest c of a nonzero x, S = sum_k floor(a_k^2 2^(2 c_k - 2C + 30))
//     as an unsigned 64-bit integer (the same whatever order the threads add in),
//     ms = RN(RN(RN(S) 2^(2C - 30)) / K), r = RN(1 / RN(sqrt(RN(ms + eps)))),
//     h = bf16(RN(RN(x r) gamma)).  An all-zero row (or one whose largest |x| is below
//     2^-40, outside the domain) gives h = 0.
//   SwiGLU: from the fp32 output of a gate+up linear, gate g = columns 0 .. K-1 and
//     up u = columns K .. 2K-1: h = bf16(RN(RN(g sg) u)), sg = RN(1 / RN(1 + e)),
//     e = e^-g by Cody and Waite's method: n = rint(RN(a log2 e)), r = a - n ln2 with
//     ln2 split into a 10-bit head and a tail (two fused multiply-adds), the degree-7
//     Taylor polynomial of e^r by Horner's rule in fused multiply-adds, times 2^n (one rounding);
//     a >= 88.72 gives +inf, a <= -87 gives 0.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "woq_device.cuh"

namespace woq {
namespace pro {

// e^a in fp32 (Cody-Waite reduction, degree-7 Taylor polynomial)
__device__ __forceinline__ float exp_cw(float a) {
  if (a >= 88.72f) return __int_as_float(0x7f800000);
  if (a <= -87.0f) return 0.0f;
  const float n = rintf(__fmul_rn(a, 0x1.715476p+0f));  // log2 e
  float r = __fmaf_rn(-n, 0x1.63p-1f, a);               // ln2 head: 0.693359375
  r = __fmaf_rn(-n, -0x1.bd0106p-13f, r);               // ln2 tail
  float p = 0x1.a01a02p-13f;                            // 1/5040
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);                 // 1/720
  p = __fmaf_rn(p, r, 0x1.111112p-7f);                  // 1/120
  p = __fmaf_rn(p, r, 0x1.555556p-5f);                  // 1/24
  p = __fmaf_rn(p, r, 0x1.555556p-3f);                  // 1/6
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  // p 2^n, rounded once: n is in [-126, 128] here, so 2^n is a normal float but for n = 128,
  // which takes two exact steps (p 2^127 is exact; doubling it rounds once)
  const int ni = (int)n;
  if (ni > 127) return __fmul_rn(__fmul_rn(p, 0x1p127f), 2.0f);
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float v) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// SwiGLU of one (gate, up) pair -> bf16 bits
__device__ __forceinline__ uint32_t swiglu_bf16(float g, float u) {
  const float e = exp_cw(-g);
  const float sg = __frcp_rn(__fadd_rn(1.0f, e));
  return f32_to_bf16_bits(__fmul_rn(__fmul_rn(g, sg), u));
}

// exponent c of a nonzero bf16 value a 2^c (a < 256); -1000 for zero
__device__ __forceinline__ int bf16_exp_c(uint32_t b16) {
  const uint32_t ef = (b16 >> 7) & 0xFFu;
  return ef ? (int)ef - 134 : ((b16 & 0x7Fu) ? -133 : -1000);
}

// a^2 2^(2c - 2C + 30) rounded down, for one bf16 value against the row exponent C (c <= C,
// so the shift is at most 30: a^2 < 2^16 times 2^sh is one 32 x 32 -> 64-bit product, and a
// negative shift leaves a 32-bit value, zero once it reaches 16)
__device__ __forceinline__ unsigned long long rms_term(uint32_t b16, int C) {
  const uint32_t ef = (b16 >> 7) & 0xFFu, f = b16 & 0x7Fu;
  const uint32_t a = ef ? 128u + f : f;
  const int c = ef ? (int)ef - 134 : -133;
  const uint32_t a2 = a * a;
  const int sh = 2 * c - 2 * C + 30;
  if (sh >= 0) return (unsigned long long)a2 * (1u << sh);
  return -sh < 16 ? (unsigned long long)(a2 >> (-sh)) : 0ull;
}

// r = RN(1 / RN(sqrt(RN(ms + eps)))) from the row's integer sum of squares
__device__ __forceinline__ float rms_rcp(unsigned long long S, int C, int K, float eps) {
  const float ms = __fdiv_rn(ldexpf(__ull2float_rn(S), 2 * C - 30), (float)K);
  return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

// h = bf16(RN(RN(x r) gamma)) of eight bf16 x against eight bf16 gamma
__device__ __forceinline__ uint4 rms_h8(uint4 x, uint4 g, float r) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, gw[4] = {g.x, g.y, g.z, g.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x0 = __uint_as_float(xw[i] << 16), x1 = __uint_as_float(xw[i] & 0xFFFF0000u);
    const float g0 = __uint_as_float(gw[i] << 16), g1 = __uint_as_float(gw[i] & 0xFFFF0000u);
    o[i] = f32_to_bf16_bits(__fmul_rn(__fmul_rn(x0, r), g0)) |
           (f32_to_bf16_bits(__fmul_rn(__fmul_rn(x1, r), g1)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// row exponent C from the bits of the row's largest |x| (held as an fp32); -1000 if zero
// or outside the domain (largest |x| below 2^-40)
__device__ __forceinline__ int rms_row_exponent(uint32_t amax_bits) {
  const int C = bf16_exp_c(amax_bits >> 16);
  return C < -47 ? -1000 : C;
}

}  // namespace pro
}  // namespace woq
