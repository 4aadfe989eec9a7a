/* CPU check of the append kernel's scale and quotient arithmetic (not the
 * oracle).
 *
 * The kernel takes s and y = RN(1/s) from a 128-entry table by the bf16
 * mantissa of the group maximum a = (1 + m/128) * 2^E: the table holds
 * s_m = fp32((1 + m/128) / 127) and RN(1/s_m), and the exponent E is added to
 * (subtracted from) their bit patterns. It forms the int8 code of x / s
 * without a division:
 *   q0 = RN(x*y), r = fma(-s, q0, x), q = fma(r, y, q0),
 *   code = low byte of bits(RN(q + 1.5*2^23)).
 * This program first checks that the table route gives the IEEE a / 127 and
 * 1 / s for every bf16 a the kernel sends that way (biased exponent >= 40),
 * then replays the per-element fp32 steps with the C library's correctly
 * rounded fmaf and compares every code with the definition: the fp32 quotient
 * x / s (IEEE division), clamped to +-127, rounded half to even. The quotient
 * check runs over every bf16 group maximum a of the listed exponents (all 128
 * mantissas), or of every exponent with a few mantissas, and every bf16 x
 * with |x| <= a, both signs. Scaling a and x by a power of two scales every
 * step exactly (no overflow or underflow in this range), so a handful of
 * exponents stands for all of them. A second part does the same for fp16
 * group scales (below). Prints "tested N bad M"; exit status 1 if M > 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16(uint32_t b) {
  uint32_t u = b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static long bad, tested;
static uint32_t tab_s[128], tab_y[128];

static float from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* s and y of group maximum a (fp32 bits) by the table route */
static void table_scale(uint32_t abits, float* s, float* y) {
  const int sh = (int)((abits >> 23) - 127) * (1 << 23);
  const uint32_t m = (abits >> 16) & 0x7fu;
  *s = from_bits(tab_s[m] + (uint32_t)sh);
  *y = from_bits(tab_y[m] - (uint32_t)sh);
}

static void check_max(uint32_t ab) {
  const volatile float a = bf16(ab);
  if ((ab >> 7) < 40) return; /* the kernel divides per element below this */
  float s, y;
  table_scale(ab << 16, &s, &y);
  for (uint32_t xb = 0; xb <= ab; ++xb) {
    for (int neg = 0; neg < 2; ++neg) {
      const volatile float x = neg ? -bf16(xb) : bf16(xb);
      float e = x / s;
      if (e > 127.0f) e = 127.0f;
      if (e < -127.0f) e = -127.0f;
      const int32_t want = (int32_t)nearbyintf(e);
      const volatile float q0 = x * y;
      const volatile float r = fmaf(-s, q0, x);
      const volatile float q = fmaf(r, y, q0);
      const volatile float t = q + 12582912.0f;
      const uint32_t code = bits(t) & 0xffu;
      ++tested;
      if (code != ((uint32_t)want & 0xffu)) {
        if (bad < 5) printf("a=%a x=%a want=%d got=%u\n", (double)a, (double)x, want, code);
        ++bad;
      }
    }
  }
}

/* The same steps with an fp16 group scale s (the pages' INT8 layout):
 * s = RN_fp16(a / 127) is a normal fp16 number, y = RN(1/s) by IEEE division,
 * and x runs over every bf16 value with |x| <= 127 s (1 + 2^-11), the largest
 * element a group with that scale can hold. The kernel sends groups whose
 * scale is an fp16 subnormal, or saturated, to the per-element division. */
static float f16(uint32_t h) {
  const int e = (int)((h >> 10) & 0x1f), m = (int)(h & 0x3ff);
  return e == 0 ? ldexpf((float)m, -24) : ldexpf((float)(1024 + m), e - 25);
}

static void check_f16_scale(uint32_t sbits) {
  const volatile float s = f16(sbits);
  const volatile float y = 1.0f / s;
  const double bound = 127.0 * (double)s * (1.0 + ldexp(1.0, -11));
  for (uint32_t xb = 0; xb < 0x7f80u; ++xb) {
    if ((double)bf16(xb) > bound) break;
    for (int neg = 0; neg < 2; ++neg) {
      const volatile float x = neg ? -bf16(xb) : bf16(xb);
      float e = x / s;
      if (e > 127.0f) e = 127.0f;
      if (e < -127.0f) e = -127.0f;
      const int32_t want = (int32_t)nearbyintf(e);
      const volatile float q0 = x * y;
      const volatile float r = fmaf(-s, q0, x);
      const volatile float q = fmaf(r, y, q0);
      const volatile float t = q + 12582912.0f;
      const uint32_t code = bits(t) & 0xffu;
      ++tested;
      if (code != ((uint32_t)want & 0xffu)) {
        if (bad < 5) printf("fp16 s=%a x=%a want=%d got=%u\n", (double)s, (double)x, want, code);
        ++bad;
      }
    }
  }
}

int main(void) {
  for (uint32_t m = 0; m < 128; ++m) {
    const volatile float sm = (1.0f + (float)m * 0.0078125f) / 127.0f;
    tab_s[m] = bits(sm);
    tab_y[m] = bits(1.0f / sm);
  }
  for (uint32_t ab = 40u << 7; ab < 0x7f80u; ++ab) {
    const volatile float a = bf16(ab);
    const float s_ieee = a / 127.0f;
    float s, y;
    table_scale(ab << 16, &s, &y);
    ++tested;
    if (bits(s) != bits(s_ieee) || bits(y) != bits(1.0f / s_ieee)) {
      if (bad < 5) printf("table a=%a s=%a want %a\n", (double)a, (double)s, (double)s_ieee);
      ++bad;
    }
  }
  static const int exps[] = {-87, -86, -60, -20, -1, 0, 1, 6, 7, 30, 100, 126, 127};
  for (unsigned i = 0; i < sizeof(exps) / sizeof(exps[0]); ++i)
    for (uint32_t m = 0; m < 128; ++m) check_max((uint32_t)(exps[i] + 127) << 7 | m);
  static const uint32_t mants[] = {0, 1, 63, 64, 126, 127};
  for (uint32_t be = 40; be < 255; ++be)
    for (unsigned i = 0; i < sizeof(mants) / sizeof(mants[0]); ++i) check_max(be << 7 | mants[i]);
  /* fp16 scales: every mantissa at exponent 0, and the smallest and largest
   * normal binades (bf16 elements down to the subnormals) */
  for (uint32_t m = 0; m < 1024; ++m) check_f16_scale(15u << 10 | m);
  for (uint32_t m = 0; m < 1024; m += 17) {
    check_f16_scale(1u << 10 | m);
    check_f16_scale(30u << 10 | m);
  }
  printf("tested %ld bad %ld\n", tested, bad);
  return bad != 0;
}
