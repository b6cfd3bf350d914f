/*
 * quotient_check.c -- checks, on the CPU, the reciprocal-based quotient that
 * the quantizer kernels use in place of an IEEE division, against the IEEE
 * division itself.  It restates the kernels' arithmetic (every operation
 * rounded once to FP32, fused multiply-adds through fmaf) and shares no code
 * with the kernels or the oracle.
 *
 * Kernel arithmetic being checked (scale s, nr = -fl32(1 / s)):
 *   one step (bf16 inputs):   Q0 = x * nr; e = fma(Q0, s, x); Q = fma(e, nr, Q0)
 *   two steps (FP32 inputs):  Q0 = x * nr; e0 = fma(Q0, s, x); Q1 = fma(e0, nr, Q0);
 *                             e1 = fma(Q1, s, x); Q = fma(e1, nr, Q1)
 * Q is the negated quotient; the kernel codes -Q.  The claims:
 *   (a) where |fl32(x / s)| >= 2^-12, -Q equals fl32(x / s) bit for bit, so
 *       the E4M3 codes agree; below that, |Q| <= 2^-10 (half the smallest
 *       E4M3 subnormal, so both code to zero) and Q has the opposite sign of
 *       x (so -Q codes to a zero of x's sign, as x / s does);
 *   (b) the same for the E5M6 cache with the bound 2^-22 and the zero
 *       threshold 2^-21 (half of its smallest subnormal 2^-20);
 *   (c) the two-step form equals fl32(x / s) for full FP32 x.
 * (a) and (b) run over every pair of a positive finite bf16 max-abs value
 * `amax` whose scale s = fl32(amax / fmt_max) is at least 2^-92 (smaller
 * scales take the kernels' exact-division path) and every bf16 x with
 * |x| <= amax, both signs.  (c) runs over a seeded sample.
 *
 * Usage: quotient_check one_step_e4m3 | one_step_e5m6 | two_step <n> |
 *                       no_step_e4m3 (the product without its correction: a
 *                       planted mistake, expected to mismatch)
 * Prints "pairs=<n> mismatches=<m>" and the first mismatches.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static uint32_t u_of(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static float one_step(float x, float s, float nr) {
  const float q0 = x * nr;
  const float e = fmaf(q0, s, x);
  return fmaf(e, nr, q0);
}

/* the first product alone, without the correction step (a planted mistake
 * that the check must catch) */
static float no_step(float x, float s, float nr) {
  (void)s;
  return x * nr;
}

static float two_step(float x, float s, float nr) {
  const float q0 = x * nr;
  const float e0 = fmaf(q0, s, x);
  const float q1 = fmaf(e0, nr, q0);
  const float e1 = fmaf(q1, s, x);
  return fmaf(e1, nr, q1);
}

static long long mismatches = 0, pairs = 0;

static int printed = 0;

static void print_mismatch(float x, float s, float got_neg, float want) {
  if (printed < 10) printf("mismatch x=%a s=%a -Q=%a x/s=%a\n", x, s, -got_neg, want);
  ++printed;
}

static void report(float x, float s, float got_neg, float want) {
  print_mismatch(x, s, got_neg, want);
  ++mismatches;
}

/* every bf16 pair for a one-step check with format maximum fmt_max, exact
 * threshold `lo` and zero threshold `zero` (amax values split over threads) */
static void check_one_step(float fmt_max, float lo, float zero, int correct) {
  const float smin = 0x1.0p-92f;
  long long n_pairs = 0, n_bad = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : n_pairs, n_bad)
  for (int ab = 1; ab < 0x7F80; ++ab) { /* positive finite bf16 amax */
    const float amax = f_of((uint32_t)ab << 16);
    const float s = amax / fmt_max;
    if (!(s >= smin)) continue;
    const float nr = -(1.0f / s);
    for (uint32_t xb = 0; xb <= (uint32_t)ab; ++xb) {
      for (int sign = 0; sign < 2; ++sign) {
        const float x = f_of((xb << 16) | (sign ? 0x80000000u : 0u));
        const float want = x / s;
        const float q = correct ? one_step(x, s, nr) : no_step(x, s, nr);
        ++n_pairs;
        int bad;
        if (fabsf(want) >= lo) {
          bad = u_of(-q) != u_of(want);
        } else {
          const int sx = (u_of(x) >> 31) & 1, sq = (u_of(q) >> 31) & 1;
          bad = !(fabsf(q) <= zero) || sx == sq;
        }
        if (bad) {
#pragma omp critical
          print_mismatch(x, s, q, want);
          ++n_bad;
        }
      }
    }
  }
  pairs += n_pairs;
  mismatches = n_bad;
}

/* splitmix64 */
static uint64_t sm_state = 0x0123456789ABCDEFull;
static uint64_t sm_next(void) {
  uint64_t z = (sm_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* n sampled FP32 pairs: amax with a random exponent in [2^-80, 2^120) and a
 * random significand, s = fl32(amax / 448); x a random FP32 value with
 * |x| <= amax (a random significand at a random exponent at most amax's,
 * plus the edge values amax and the largest float below it) */
static void check_two_step(long long n) {
  for (long long i = 0; i < n; ++i) {
    const uint64_t r = sm_next();
    const uint32_t ae = 47u + (uint32_t)(r % 200u); /* biased exponent 47..246 */
    const uint32_t am = (uint32_t)(r >> 8) & 0x7FFFFFu;
    const float amax = f_of((ae << 23) | am);
    const float s = amax / 448.0f;
    if (!(s >= 0x1.0p-92f)) continue;
    const float nr = -(1.0f / s);
    const uint64_t r2 = sm_next();
    float x;
    const uint32_t kind = (uint32_t)(r2 & 15u);
    if (kind == 0) {
      x = amax;
    } else if (kind == 1) {
      x = nextafterf(amax, 0.0f);
    } else {
      const uint32_t span = 40u;
      const uint32_t d = (uint32_t)((r2 >> 4) % span);
      const uint32_t xe = ae > d ? ae - d : 1u;
      x = f_of((xe << 23) | ((uint32_t)(r2 >> 16) & 0x7FFFFFu));
      if (x > amax) x = amax;
    }
    if (r2 >> 63) x = -x;
    const float want = x / s;
    const float q = two_step(x, s, nr);
    ++pairs;
    if (fabsf(want) >= 0x1.0p-11f) {
      if (u_of(-q) != u_of(want)) report(x, s, q, want);
    } else {
      const int sx = (u_of(x) >> 31) & 1, sq = (u_of(q) >> 31) & 1;
      if (!(fabsf(q) <= 0x1.0p-10f) || sx == sq) report(x, s, q, want);
    }
  }
}

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  if (!strcmp(argv[1], "one_step_e4m3"))
    check_one_step(448.0f, 0x1.0p-12f, 0x1.0p-10f, 1);
  else if (!strcmp(argv[1], "one_step_e5m6"))
    check_one_step(65024.0f, 0x1.0p-22f, 0x1.0p-21f, 1);
  else if (!strcmp(argv[1], "no_step_e4m3"))
    check_one_step(448.0f, 0x1.0p-12f, 0x1.0p-10f, 0);
  else if (!strcmp(argv[1], "two_step") && argc >= 3)
    check_two_step(atoll(argv[2]));
  else
    return 2;
  printf("pairs=%lld mismatches=%lld\n", pairs, mismatches);
  return 0;
}
