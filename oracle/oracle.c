/*
 * CPU oracle for the weight-only-quantised skinny linear (W4A8 / W6A8).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously correct
 * restatement of what the skinny linear computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or helper with the CUDA library, and it never reads the
 * library's packed device layout: it works on the canonical checkpoint layout.
 *
 * What it follows ("Doubling LLM token rates in ComfyUI", blog.comfy.org):
 *   - section "What is the bottleneck?": the op is a dense N x K weight matrix
 *     times a skinny M x K activation (M = 1 for one token, a few rows for
 *     multi-token-prediction verification);
 *   - section "Optimizing the Linear Kernel": W4A8 / W6A8 checkpoints carry
 *     4- or 6-bit weights with one scale per group of weights, and the
 *     activation is quantised to 8 bits before an integer matrix-vector
 *     product (dp4a or int8 MMA, i.e. int8 x int8 -> int32 dot products).
 *
 * The pages give no formulas, bit layouts or rounding rules.  The readings
 * used here (each one is also listed with the design notes):
 *   R1  weights are N x K (output x input); groups are 128 consecutive k of
 *       one output row, starting at k = 0; K % 128 == 0;
 *   R2  int4 weights are two's complement in [-8, 7], two per byte along K,
 *       the low nibble holding the even k;
 *   R3  int6 weights are two's complement in [-32, 31], four per three bytes
 *       along K, read as a little-endian 24-bit word with value i in bits
 *       6i .. 6i+5;
 *   R4  one fp16 scale per (row, group), symmetric (no zero point): the real
 *       weight is q * scale;
 *   R5  activation quantisation is per row (token): amax = max |x| in fp32,
 *       scale = amax / 127 (one IEEE fp32 division), q = round-half-even of
 *       the IEEE fp32 quotient x / scale, clamped to [-127, 127]; an all-zero
 *       row gives scale 0 and q 0;
 *   R6  per group g: d = sum over the group of q_w * q_a (exact integer);
 *       term = (fp32(d) * scale_w) * scale_a, two fp32 roundings in that
 *       order; y = sum over g of the terms, here summed in fp64 in g order
 *       and rounded once to fp32;
 *   R7  non-finite activations are outside the domain (rejected here);
 *       subnormals are kept (no flush to zero).
 *   R11 (prologue fusion, RMSNorm) h = bf16(RN(RN(x * r) * gamma)) per element,
 *       r = RN(1 / RN(sqrt(RN(RN(ms) + eps)))), where the mean of squares ms is
 *       formed from exact squares: a bf16 x is a 2^c with a an integer < 256, so
 *       x^2 = a^2 2^(2c); the row sum S = sum_k floor(a_k^2 2^(2 c_k - 2 C + 30))
 *       2^(2C - 30) (C the largest c of a nonzero x of the row; an unsigned 64-bit
 *       integer sum, independent of the order of summation), ms = RN(RN(S) / K).
 *       An all-zero row gives h = 0.  Rows whose largest |x| is below 2^-40 are
 *       outside the domain;
 *   R12 (prologue fusion, SwiGLU) input: the fp32 [M][2K] output of a gate+up
 *       linear (gate = columns 0 .. K-1, up = K .. 2K-1); h = bf16(RN(RN(g * sg)
 *       * u)), sg = RN(1 / RN(1 + e)), e = exp(-g) evaluated in fp32 by the
 *       Cody-Waite method: n = rint(RN(a log2 e)), r = a - n ln2 with ln2 split in
 *       two constants (two fused multiply-adds), the degree-7 Taylor polynomial of
 *       e^r by Horner's rule with fused multiply-adds, scaled by 2^n; a >= 88.72
 *       gives +inf and a <= -87 gives 0;
 *   R13 both fusions quantise the bf16 h exactly as R5 quantises x.
 *
 * The fp16 and bf16 decoders are written from the IEEE 754 encodings.
 * Build: plain C11, no -ffast-math, -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* status codes of the oracle's own entry points */
#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE 1
#define ORACLE_ERR_NONFINITE 2
#define ORACLE_ERR_RANGE 3
#define ORACLE_ERR_BITS 4

/* ------------------------------------------------------------------------ */
/* IEEE 754 decoders                                                         */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float oracle_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^(1-15) */
  } else if (e == 31) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
  }
  return (float)(sign ? -v : v);
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
float oracle_bf16_to_f32(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xFF;
  int f = b & 0x7F;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133); /* subnormal: f * 2^-7 * 2^(1-127) */
  } else if (e == 255) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
  }
  return (float)(sign ? -v : v);
}

/* ------------------------------------------------------------------------ */
/* canonical weight decoding (R2, R3)                                        */
/* ------------------------------------------------------------------------ */

/* weight (n, k) of a canonical int4 matrix with K columns */
int oracle_w4_at(const uint8_t* w4, int K, int n, int k) {
  uint8_t byte = w4[(size_t)n * (size_t)(K / 2) + (size_t)(k / 2)];
  int nib = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  return nib >= 8 ? nib - 16 : nib;
}

/* weight (n, k) of a canonical int6 matrix with K columns */
int oracle_w6_at(const uint8_t* w6, int K, int n, int k) {
  const uint8_t* p = w6 + (size_t)n * (size_t)(K / 4 * 3) + (size_t)(k / 4) * 3;
  uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16);
  int field = (int)((word >> (6 * (k % 4))) & 0x3F);
  return field >= 32 ? field - 64 : field;
}

static int weight_at(int bits, const uint8_t* w, int K, int n, int k) {
  return bits == 4 ? oracle_w4_at(w, K, n, k) : oracle_w6_at(w, K, n, k);
}

/* unpack a whole canonical matrix into one int8 per weight, row-major N x K */
int oracle_unpack_weights(int bits, const uint8_t* w, int N, int K, int8_t* out) {
  if (bits != 4 && bits != 6) return ORACLE_ERR_BITS;
  if (N < 0 || K < 0 || K % 128 != 0) return ORACLE_ERR_SHAPE;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) out[(size_t)n * K + k] = (int8_t)weight_at(bits, w, K, n, k);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* activation quantisation (R5)                                              */
/* ------------------------------------------------------------------------ */

int oracle_act_quant(const uint16_t* x_bf16, int M, int K, int8_t* q, float* ascale) {
  if (M < 0 || K < 0) return ORACLE_ERR_SHAPE;
  for (int m = 0; m < M; ++m) {
    const uint16_t* xr = x_bf16 + (size_t)m * K;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float v = oracle_bf16_to_f32(xr[k]);
      if (!isfinite(v)) return ORACLE_ERR_NONFINITE;
      float a = fabsf(v);
      if (a > amax) amax = a;
    }
    float s = amax / 127.0f; /* one IEEE fp32 division */
    ascale[m] = s;
    for (int k = 0; k < K; ++k) {
      int qi = 0;
      if (s != 0.0f) {
        float t = oracle_bf16_to_f32(xr[k]) / s; /* IEEE fp32 quotient */
        float r = nearbyintf(t);                 /* default mode: to nearest, ties to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        qi = (int)r;
      }
      q[(size_t)m * K + k] = (int8_t)qi;
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* per-group integer dot products (R6, first half)                           */
/* ------------------------------------------------------------------------ */

/* dots[(m * N + n) * G + g] = sum_{k in group g} w(n, k) * q(m, k), exact */
int oracle_group_dots(int bits, const uint8_t* w, int N, int K, const int8_t* q, int M, int32_t* dots) {
  if (bits != 4 && bits != 6) return ORACLE_ERR_BITS;
  if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return ORACLE_ERR_SHAPE;
  const int G = K / 128;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n)
      for (int g = 0; g < G; ++g) {
        int64_t s = 0;
        for (int k = g * 128; k < g * 128 + 128; ++k)
          s += (int64_t)weight_at(bits, w, K, n, k) * (int64_t)q[(size_t)m * K + k];
        if (s >= (1 << 24) || s <= -(1 << 24)) return ORACLE_ERR_RANGE; /* must be exact in fp32 */
        dots[((size_t)m * N + n) * G + g] = (int32_t)s;
      }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* the linear (R6)                                                           */
/* ------------------------------------------------------------------------ */

/* y[m * N + n] = sum_g (fp32(d) * ws[n, g]) * as[m]; S[m * N + n] = sum_g |term|
 * (S may be NULL).  wscale_f16 is N x G row-major fp16 bit patterns. */
int oracle_gemv(int bits, const uint8_t* w, const uint16_t* wscale_f16, int N, int K, const int8_t* q,
                const float* ascale, int M, float* y, double* S) {
  if (bits != 4 && bits != 6) return ORACLE_ERR_BITS;
  if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return ORACLE_ERR_SHAPE;
  const int G = K / 128;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      double sum = 0.0, sabs = 0.0;
      for (int g = 0; g < G; ++g) {
        int64_t d = 0;
        for (int k = g * 128; k < g * 128 + 128; ++k)
          d += (int64_t)weight_at(bits, w, K, n, k) * (int64_t)q[(size_t)m * K + k];
        if (d >= (1 << 24) || d <= -(1 << 24)) return ORACLE_ERR_RANGE;
        float ws = oracle_f16_to_f32(wscale_f16[(size_t)n * G + g]);
        float t = (float)d * ws; /* first fp32 rounding */
        t = t * ascale[m];       /* second fp32 rounding */
        sum += (double)t;
        sabs += fabs((double)t);
      }
      y[(size_t)m * N + n] = (float)sum;
      if (S) S[(size_t)m * N + n] = sabs;
    }
  return ORACLE_OK;
}

/* act_quant followed by the linear: the whole op from bf16 activations. */
int oracle_linear_bf16(int bits, const uint8_t* w, const uint16_t* wscale_f16, int N, int K, const uint16_t* x_bf16,
                       int M, float* y, double* S) {
  if (M < 0 || K < 0) return ORACLE_ERR_SHAPE;
  int8_t* q = (int8_t*)malloc((size_t)M * (size_t)K + 1);
  float* as = (float*)malloc((size_t)M * sizeof(float) + 1);
  if (!q || !as) {
    free(q);
    free(as);
    return ORACLE_ERR_SHAPE;
  }
  int rc = oracle_act_quant(x_bf16, M, K, q, as);
  if (rc == ORACLE_OK) rc = oracle_gemv(bits, w, wscale_f16, N, K, q, as, M, y, S);
  free(q);
  free(as);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* prologue fusions (R11 - R13; section "Optimizing the Linear Kernel": the  */
/* RMSNorm or SwiGLU before a linear is folded into its input quantisation)  */
/* ------------------------------------------------------------------------ */

/* fp32 -> bf16 bit pattern, round to nearest, ties to even (finite inputs) */
uint16_t oracle_f32_to_bf16(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  const uint32_t keep = u >> 16, rem = u & 0xFFFFu;
  uint32_t r = keep;
  if (rem > 0x8000u || (rem == 0x8000u && (keep & 1u))) r = keep + 1u;
  return (uint16_t)r;
}

/* e^a in fp32 by Cody-Waite argument reduction and a degree-7 Taylor polynomial */
float oracle_exp_cw(float a) {
  if (a >= 88.72f) return INFINITY;
  if (a <= -87.0f) return 0.0f;
  const float n = rintf(a * 1.44269504f);
  float r = fmaf(-n, 0.693359375f, a);
  r = fmaf(-n, -2.12194440e-4f, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return ldexpf(p, (int)n);
}

/* a bf16 value as a 2^c with 0 <= a < 256: returns a, writes c */
static uint32_t bf16_int_exp(uint16_t b, int* c) {
  const uint32_t ef = (b >> 7) & 0xFFu, f = b & 0x7Fu;
  if (ef == 0) {
    *c = -133;
    return f;
  }
  *c = (int)ef - 134;
  return 128u + f;
}

int oracle_rmsnorm_bf16(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, uint16_t* h) {
  if (M < 0 || K < 0) return ORACLE_ERR_SHAPE;
  for (int m = 0; m < M; ++m) {
    const uint16_t* xr = x + (size_t)m * K;
    uint16_t* hr = h + (size_t)m * K;
    int C = -1000;
    for (int k = 0; k < K; ++k) {
      if (!isfinite(oracle_bf16_to_f32(xr[k]))) return ORACLE_ERR_NONFINITE;
      int c;
      if (bf16_int_exp(xr[k], &c) != 0 && c > C) C = c;
    }
    if (C == -1000) { /* all zero */
      for (int k = 0; k < K; ++k) hr[k] = 0;
      continue;
    }
    if (C < -47) return ORACLE_ERR_RANGE; /* largest |x| below 2^-40 */
    uint64_t S = 0;
    for (int k = 0; k < K; ++k) {
      int c;
      const uint64_t a = bf16_int_exp(xr[k], &c);
      const int sh = 2 * c - 2 * C + 30; /* a^2 2^(2c) in units of 2^(2C - 30) */
      if (a == 0) continue;
      if (sh >= 0)
        S += (a * a) << sh;
      else if (sh > -64)
        S += (a * a) >> (-sh);
    }
    const float s1 = (float)S; /* round to nearest */
    const float ms = ldexpf(s1, 2 * C - 30) / (float)K;
    const float sd = sqrtf(ms + eps);
    const float r = 1.0f / sd;
    for (int k = 0; k < K; ++k) {
      const float xr_k = oracle_bf16_to_f32(xr[k]) * r;
      hr[k] = oracle_f32_to_bf16(xr_k * oracle_bf16_to_f32(gamma[k]));
    }
  }
  return ORACLE_OK;
}

int oracle_swiglu_bf16(const float* gu, int M, int K, uint16_t* h) {
  if (M < 0 || K < 0) return ORACLE_ERR_SHAPE;
  for (int m = 0; m < M; ++m) {
    const float* g = gu + (size_t)m * 2 * K;
    const float* u = g + K;
    for (int k = 0; k < K; ++k) {
      if (!isfinite(g[k]) || !isfinite(u[k])) return ORACLE_ERR_NONFINITE;
      const float e = oracle_exp_cw(-g[k]);
      const float sg = 1.0f / (1.0f + e);
      const float si = g[k] * sg;
      h[(size_t)m * K + k] = oracle_f32_to_bf16(si * u[k]);
    }
  }
  return ORACLE_OK;
}
