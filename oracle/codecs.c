/*
 * codecs.c -- number formats of the caches (test infrastructure; see
 * bsp_oracle.h).
 *
 * The formats are the ones the pages name: e4m3 for the fp8 K/V cache and the
 * e4m3 query ([ATOM-2962] commit "... the kernel writes the unit-scale
 * saturating cast"), and MXFP4 = e2m1 data with one e8m0 scale per 32
 * elements ([ATOM-2962] PR description, "FP4 index cache").  Each encoder is
 * written as "round to the nearest representable value, ties to the even
 * code, then saturate", computed on exact fp64 values, not by bit tricks.
 */
#include "bsp_oracle.h"

#include <math.h>
#include <string.h>

/* e4m3 (OCP FP8 E4M3FN): bias 7, 3 mantissa bits, subnormals m/8 * 2^-6,
 * largest finite 448, codes 0x7F/0xFF are NaN, no infinity. */
double orc_e4m3_decode(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

uint8_t orc_e4m3_encode(float xf) {
  double x = (double)xf;
  uint8_t sign = signbit(xf) ? 0x80 : 0x00;
  double a = fabs(x);
  if (isnan(xf)) return (uint8_t)(sign | 0x7F);
  /* quantum of the binade holding a; below 2^-6 the spacing is 2^-9 */
  int e;
  if (a < ldexp(1.0, -6)) {
    e = -6;
  } else {
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;             /* a in [2^e, 2^(e+1)) */
  }
  double quantum = ldexp(1.0, e - 3);
  double q = nearbyint(a / quantum); /* default rounding mode: ties to even */
  double v = q * quantum;
  if (v > 448.0) v = 448.0; /* satfinite */
  /* encode the (now representable) magnitude v */
  if (v == 0.0) return sign;
  int ee;
  if (v < ldexp(1.0, -6)) {
    int m = (int)(v / ldexp(1.0, -9));
    return (uint8_t)(sign | m);
  }
  (void)frexp(v, &ee);
  ee -= 1;
  int m = (int)((v / ldexp(1.0, ee) - 1.0) * 8.0);
  return (uint8_t)(sign | ((ee + 7) << 3) | m);
}

/* e2m1: sign bit 3, two exponent bits (bias 1), one mantissa bit.  The eight
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t nib) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[nib & 7];
  return (nib & 8) ? -v : v;
}

uint8_t orc_e2m1_encode(double x) {
  uint8_t sign = signbit(x) ? 8 : 0;
  double a = fabs(x);
  if (isnan(x)) return (uint8_t)(sign | 7); /* no NaN code; never produced here */
  double quantum = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  double v = nearbyint(a / quantum) * quantum;
  if (v > 6.0) v = 6.0;
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  for (int c = 0; c < 8; ++c)
    if (mag[c] == v) return (uint8_t)(sign | c);
  return (uint8_t)(sign | 7);
}

double orc_e8m0_decode(uint8_t b) { return ldexp(1.0, (int)b - 127); }

float orc_bf16_decode(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t orc_bf16_encode(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return (uint16_t)((u >> 16) | 0x40);
  /* round to nearest, ties to even, on the 16 dropped bits */
  uint32_t lower = u & 0xFFFFu, upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;
  return (uint16_t)upper;
}

/* MXFP4 shared exponent.  Reading (the pages give no rule): the OCP MX v1.0
 * choice, shared_exp = floor(log2(amax)) - emax(e2m1), emax(e2m1) = 2, clamped
 * to the e8m0 range; an all-zero group gets the smallest scale.  floor(log2)
 * is taken exactly from frexp. */
uint8_t orc_mx_scale_byte(const float* x, int n) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i)
    if (fabs((double)x[i]) > amax) amax = fabs((double)x[i]);
  int e;
  if (amax == 0.0) {
    e = -127;
  } else {
    int ex;
    (void)frexp(amax, &ex); /* amax in [2^(ex-1), 2^ex) */
    e = (ex - 1) - 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
  }
  return (uint8_t)(e + 127);
}

void orc_cast_e4m3(const uint16_t* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(orc_bf16_decode(x[i]));
}
