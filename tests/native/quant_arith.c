/* Host restatement of the two division-free steps the GPU quantizer uses
 * (the correctly rounded quotient amax/127 and reciprocal 1/d), checked here
 * against IEEE single-precision division.  Only IEEE float multiplies and
 * fmas appear, so the host computes the same bits as the device.
 *
 *   quant_arith           run every check, print one line per check, exit 1
 *                         on any mismatch
 *
 * Checks: the quotient for every significand at every exponent of the
 * sample below and every subnormal; the reciprocal for every subnormal d and
 * every significand at the exponents below (both methods scale exactly with
 * the exponent between those ranges); the reciprocal's special values. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* a / 127 for a >= 0: estimate q0 = a * RN(1/127), exact remainder by fma,
 * one correction (Markstein 1990). */
static float div127_rn(float a) {
  const float r = 0x1.020408p-7f;
  const float q0 = a * r;
  const float rem = fmaf(-q0, 127.0f, a);
  const float q1 = fmaf(rem, r, q0);
  return (a <= 3.40282347e38f) ? q1 : a;
}

/* 1/d for normal d with a normal reciprocal: bit-pattern estimate, four
 * Newton-Raphson steps with fma, one ulp up for an all-ones significand. */
static float rcp_rn_normal(float d) {
  float y = f_of(0x7EF00000u - u_of(d));
  for (int k = 0; k < 4; ++k) {
    const float e = fmaf(-d, y, 1.0f);
    y = fmaf(y, e, y);
  }
  return ((u_of(d) & 0x7FFFFFu) == 0x7FFFFFu) ? f_of(u_of(y) + 1u) : y;
}

static float rcp_rn(float d) {
  const int sub = d < 0x1p-126f;
  const float ds = sub ? d * 0x1p24f : d;
  const float ys = rcp_rn_normal(ds);
  const float y = sub ? ys * 0x1p24f : ys;
  return (d == 0.0f || d > 3.40282347e38f) ? 0.0f : y;
}

static int report(const char* what, uint64_t bad, uint64_t n) {
  printf("%s: %llu of %llu differ\n", what, (unsigned long long)bad, (unsigned long long)n);
  return bad != 0;
}

int main(void) {
  int fail = 0;
  /* exponents (unbiased) whose every significand is checked */
  static const int div_exps[] = {-126, -125, -124, -123, -122, -121, -120, -119, -118, -117,
                                 -1, 0, 1, 64, 126, 127};
  static const int rcp_exps[] = {-126, -125, -124, -123, -122, -121, -120, -1, 0, 1, 60,
                                 119, 120, 121};
  uint64_t bad = 0, n = 0;
  for (uint32_t u = 0; u < 0x00800000u; ++u, ++n)  /* subnormals and zero */
    bad += u_of(div127_rn(f_of(u))) != u_of(f_of(u) / 127.0f);
  for (unsigned i = 0; i < sizeof div_exps / sizeof div_exps[0]; ++i) {
    const uint32_t base = (uint32_t)(div_exps[i] + 127) << 23;
    for (uint32_t m = 0; m < 0x00800000u; ++m, ++n)
      bad += u_of(div127_rn(f_of(base | m))) != u_of(f_of(base | m) / 127.0f);
  }
  fail |= report("div127_rn", bad, n);

  bad = 0;
  n = 0;
  for (uint32_t u = 1; u < 0x00800000u; ++u, ++n)  /* subnormal d */
    bad += u_of(rcp_rn(f_of(u))) != u_of(1.0f / f_of(u));
  for (unsigned i = 0; i < sizeof rcp_exps / sizeof rcp_exps[0]; ++i) {
    const uint32_t base = (uint32_t)(rcp_exps[i] + 127) << 23;
    for (uint32_t m = 0; m < 0x00800000u; ++m, ++n)
      bad += u_of(rcp_rn(f_of(base | m))) != u_of(1.0f / f_of(base | m));
  }
  fail |= report("rcp_rn", bad, n);

  bad = (rcp_rn(0.0f) != 0.0f) + (rcp_rn(INFINITY) != 0.0f) + !isnan(rcp_rn(NAN)) +
        (div127_rn(INFINITY) != INFINITY) + !isnan(div127_rn(NAN));
  fail |= report("special values", bad, 5);
  return fail;
}
