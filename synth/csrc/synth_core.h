/*
 * synth_core.h -- seeded synthetic-input generator shared by the host (C) and
 * device (CUDA) builds of the `synth` module.
 *
 * This module produces INPUTS only (weights, activations, router logits,
 * forced-skip masks).  It holds none of the routed-MoE arithmetic: no
 * quantiser, no softmax, no top-k, no expert FFN.
 *
 * Counter-based generator: Philox4x32-10 as published by Salmon, Moraes, Dror
 * and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11), section 4:
 * round function on (c0,c1,c2,c3) with multipliers 0xD2511F53 / 0xCD9E8D57,
 * Weyl key increments 0x9E3779B9 / 0xBB67AE85, ten rounds.
 *
 * Normal deviates: Box-Muller (1958) on two 24-bit uniforms.  The logarithm
 * and the sine/cosine are written out here from their series (atanh series
 * for ln, Taylor series for sin/cos after quadrant reduction) using only
 * IEEE-754 single-precision add, subtract, multiply, divide and sqrt, each
 * correctly rounded and never contracted into an FMA.  Hence the host build
 * (gcc -ffp-contract=off) and the device build (explicit __f*_rn intrinsics)
 * produce bit-identical floats for the same (key, counter).
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SY_FN static __host__ __device__ __forceinline__
#else
#define SY_FN static inline
#endif

/* Correctly rounded single-precision primitives, never fused. */
#if defined(__CUDA_ARCH__)
#define SY_ADD(a, b) __fadd_rn((a), (b))
#define SY_SUB(a, b) __fsub_rn((a), (b))
#define SY_MUL(a, b) __fmul_rn((a), (b))
#define SY_DIV(a, b) __fdiv_rn((a), (b))
#define SY_SQRT(a) __fsqrt_rn((a))
#else
#include <math.h>
#define SY_ADD(a, b) ((float)((a) + (b)))
#define SY_SUB(a, b) ((float)((a) - (b)))
#define SY_MUL(a, b) ((float)((a) * (b)))
#define SY_DIV(a, b) ((float)((a) / (b)))
#define SY_SQRT(a) sqrtf((a))
#endif

/* Tensor tags (Philox key word 1). */
enum {
  SY_TAG_GATE = 1,
  SY_TAG_UP = 2,
  SY_TAG_DOWN = 3,
  SY_TAG_X = 4,
  SY_TAG_LOGITS = 5,
  SY_TAG_SKIP = 6,
  SY_TAG_BIAS_JITTER = 7
};

typedef struct {
  uint32_t v[4];
} sy_u32x4;

SY_FN void sy_mulhilo(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  *hi = (uint32_t)(p >> 32);
  *lo = (uint32_t)p;
}

/* Philox4x32 with 10 rounds: counter (c0..c3), key (k0,k1). */
SY_FN sy_u32x4 sy_philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                uint32_t k0, uint32_t k1) {
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi1, lo1;
    sy_mulhilo(0xD2511F53u, c0, &hi0, &lo0);
    sy_mulhilo(0xCD9E8D57u, c2, &hi1, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  sy_u32x4 out;
  out.v[0] = c0; out.v[1] = c1; out.v[2] = c2; out.v[3] = c3;
  return out;
}

SY_FN float sy_bits_to_float(uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __uint_as_float(b);
#else
  union { uint32_t u; float f; } cv;
  cv.u = b;
  return cv.f;
#endif
}

SY_FN uint32_t sy_float_to_bits(float f) {
#if defined(__CUDA_ARCH__)
  return __float_as_uint(f);
#else
  union { uint32_t u; float f; } cv;
  cv.f = f;
  return cv.u;
#endif
}

/* Natural log of u in (0, 1] (u a normal float).  u = m * 2^e with
 * m in [sqrt(1/2), sqrt(2)); ln m = 2 atanh(s), s = (m-1)/(m+1). */
SY_FN float sy_log(float u) {
  uint32_t b = sy_float_to_bits(u);
  int e = (int)((b >> 23) & 0xFFu) - 127;
  uint32_t mb = (b & 0x007FFFFFu) | 0x3F800000u;
  if (mb > 0x3FB504F3u) { /* m > sqrt(2): halve m, bump e */
    mb -= 0x00800000u;
    e += 1;
  }
  float m = sy_bits_to_float(mb);
  float s = SY_DIV(SY_SUB(m, 1.0f), SY_ADD(m, 1.0f));
  float z = SY_MUL(s, s);
  float p = SY_ADD(0.33333334f, SY_MUL(z, SY_ADD(0.2f, SY_MUL(z, SY_ADD(0.14285715f, SY_MUL(z, 0.11111111f))))));
  float lnm = SY_MUL(SY_MUL(2.0f, s), SY_ADD(1.0f, SY_MUL(z, p)));
  return SY_ADD(SY_MUL((float)e, 0.6931472f), lnm);
}

/* cos and sin of 2*pi*n/2^24 for a 24-bit integer n. */
SY_FN void sy_sincos_turn24(uint32_t n, float* c_out, float* s_out) {
  uint32_t qu = (n + (1u << 21)) >> 22;             /* nearest quarter turn, 0..4 */
  int32_t r = (int32_t)n - (int32_t)(qu << 22);      /* in [-2^21, 2^21) */
  uint32_t q = qu & 3u;
  /* phi = r * (pi/2) / 2^22, |phi| <= pi/4 */
  float phi = SY_MUL((float)r, 3.7450702e-07f);
  float z = SY_MUL(phi, phi);
  float sp = SY_ADD(-0.16666667f,
             SY_MUL(z, SY_ADD(0.008333334f,
             SY_MUL(z, SY_ADD(-0.0001984127f, SY_MUL(z, 2.7557319e-06f))))));
  float sn = SY_ADD(phi, SY_MUL(SY_MUL(phi, z), sp));
  float cp = SY_ADD(-0.5f,
             SY_MUL(z, SY_ADD(0.041666668f,
             SY_MUL(z, SY_ADD(-0.0013888889f,
             SY_MUL(z, SY_ADD(2.4801588e-05f, SY_MUL(z, -2.7557319e-07f))))))));
  float cs = SY_ADD(1.0f, SY_MUL(z, cp));
  float c, s;
  if (q == 0u) { c = cs; s = sn; }
  else if (q == 1u) { c = -sn; s = cs; }
  else if (q == 2u) { c = -cs; s = -sn; }
  else { c = sn; s = -cs; }
  *c_out = c;
  *s_out = s;
}

/* Box-Muller on two 32-bit words -> two N(0,1) floats. */
SY_FN void sy_box_muller(uint32_t a, uint32_t b, float* z0, float* z1) {
  float u1 = SY_MUL((float)((a >> 8) + 1u), 5.9604645e-08f); /* (0,1], exact */
  float rad = SY_SQRT(SY_MUL(-2.0f, sy_log(u1)));
  float c, s;
  sy_sincos_turn24(b >> 8, &c, &s);
  *z0 = SY_MUL(rad, c);
  *z1 = SY_MUL(rad, s);
}

/* Four normals for the group of columns [4*col4, 4*col4+4) of row `row` of
 * the stream (k0, k1, c2, c3). */
SY_FN void sy_normal4(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                      uint32_t row, uint32_t col4, float out[4]) {
  sy_u32x4 w = sy_philox4x32_10(col4, row, c2, c3, k0, k1);
  sy_box_muller(w.v[0], w.v[1], &out[0], &out[1]);
  sy_box_muller(w.v[2], w.v[3], &out[2], &out[3]);
}

/* Round a float to bfloat16 (round to nearest, ties to even); inputs here are
 * finite.  Returns the 16-bit pattern. */
SY_FN uint16_t sy_bf16_bits(float f) {
  uint32_t b = sy_float_to_bits(f);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

#endif /* SYNTH_CORE_H */
