/* CPU check of the rk8v4 scale rounding (not the oracle).
 *
 * The rk8v4 append kernel forms a group scale as __float2half_rn(__fdiv_rn(a, c)):
 * the IEEE fp32 quotient of the group maximum a by c (c = 127 for keys, 7 for
 * values), rounded again to fp16. The oracle forms RN_fp16 of the fp64
 * quotient. Both equal the correctly rounded fp16 quotient when a / c is never
 * an fp16 rounding midpoint and the first rounding never reaches one; this
 * program checks that the two routes give the same fp16 value for
 *   values: every positive finite bf16 a, c = 7;
 *   keys:   every fp32 a (all 2^23 mantissas) of the binary exponents -40 .. 30
 *           (a / 127 from below the fp16 subnormal range to past its maximum),
 *           c = 127;
 * using host IEEE fp32 division and its own round-to-fp16 (ties to even, the
 * subnormal quantum 2^-24, overflow to infinity). Prints "tested N bad M";
 * exit status 1 if M > 0.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

/* x >= 0 rounded to the nearest fp16 value, ties to even; INFINITY past 65504 */
static double round_f16(double x) {
  if (x == 0.0) return 0.0;
  int e;
  frexp(x, &e); /* x = m 2^e, 0.5 <= m < 1: leading bit 2^(e-1) */
  double r;
  if (e - 1 < -14) r = nearbyint(ldexp(x, 24)) * ldexp(1.0, -24);
  else r = ldexp(nearbyint(ldexp(x, 11 - e)), e - 11);
  return r > 65504.0 ? INFINITY : r;
}

static long tested, bad;

static void check(float a, float c) {
  const float q32 = a / c; /* IEEE fp32 quotient */
  const double kernel = round_f16((double)q32);
  const double oracle = round_f16((double)a / (double)c);
  ++tested;
  if (kernel != oracle) {
    if (bad < 10) printf("mismatch a=%a c=%g kernel=%a oracle=%a\n", (double)a, (double)c, kernel, oracle);
    ++bad;
  }
}

int main(void) {
  fesetround(FE_TONEAREST);
  /* values: every positive finite bf16 */
  for (uint32_t b = 1; b < 0x7f80u; ++b) {
    const uint32_t u = b << 16;
    float a;
    memcpy(&a, &u, 4);
    check(a, 7.0f);
  }
  /* keys: every fp32 mantissa of each exponent */
  for (int ex = -40; ex <= 30; ++ex)
    for (uint32_t m = 0; m < (1u << 23); ++m) {
      const uint32_t u = ((uint32_t)(ex + 127) << 23) | m;
      float a;
      memcpy(&a, &u, 4);
      check(a, 127.0f);
    }
  printf("tested %ld bad %ld\n", tested, bad);
  return bad ? 1 : 0;
}
