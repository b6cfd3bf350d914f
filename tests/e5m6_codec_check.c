/*
 * e5m6_codec_check.c -- checks, on the CPU, the bit arithmetic that the
 * quantizer kernels use for the 12-bit E5M6 activation cache, against the
 * format's definition computed in double precision.  It restates the
 * kernels' operations and shares no code with the kernels or the oracle.
 *
 * The format (the cache's reading of the page, which is silent on it):
 * sign, 5 exponent bits with bias 15, 6 mantissa bits; exponent 0 holds the
 * subnormals m * 2^-20, exponent 31 Inf/NaN; values are rounded to nearest
 * with ties to even, saturated at 65024 (code 0x7BF, Inf included), and a
 * NaN codes to 0x7FF.
 *
 * Modes (each prints "pairs=<n> mismatches=<m>" last):
 *   fast     the fast-path encoder of a negated quotient q = -x/s (finite,
 *            |q| below 65280, the midpoint above 65024; the code is that of
 *            -q): an integer add that rounds and rebiases, and a fused
 *            multiply-add for the subnormal multiple of 2^-20; every FP32
 *            pattern of that range, both signs;
 *   general  the encoder of the exact-division path (NaN, saturation,
 *            subnormals by an exact scaling and a round), every FP32 pattern;
 *   decode   the decoder: two codes shifted into one IEEE f16x2 word and
 *            converted, for every code at each of the four positions of a
 *            48-bit group, with seeded codes around it;
 *   pack     eight codes packed into three little-endian words, against bit
 *            by bit placement, on a seeded sample;
 *   fast_nocarry  the fast encoder with the rounding increment dropped (a
 *            planted mistake, expected to mismatch).
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

/* The definition: code of y, from its value in double precision. */
static uint32_t code_def(float y) {
  if (isnan(y)) return 0x7FFu;
  const uint32_t sign = (u_of(y) >> 31) ? 0x800u : 0u;
  const double m = fabs((double)y);
  if (m >= 65024.0) return sign | 0x7BFu;
  if (m < 0x1p-14) return sign | (uint32_t)rint(m * 0x1p20); /* 0 .. 64; 64 is 2^-14 */
  int ex;
  const double f = frexp(m, &ex); /* m = f 2^ex, f in [0.5, 1) */
  int e = ex - 1;
  double k = rint((2.0 * f - 1.0) * 64.0); /* exact product, rounded to even */
  if (k == 64.0) {
    k = 0.0;
    ++e;
  }
  return sign | ((uint32_t)(e + 15) << 6) | (uint32_t)k;
}

/* --- the kernels' arithmetic, restated -------------------------------- */

static uint32_t mag_normal(uint32_t a, int carry) {
  return (a + (carry ? ((a >> 17) & 1u) : 0u) + (0xFFFFu - (7168u << 17))) >> 17;
}

/* fast path, negated quotient bits ux */
static uint32_t code_fast(uint32_t ux, int carry) {
  const uint32_t a = ux & 0x7FFFFFFFu;
  const uint32_t sub = u_of(fmaf(f_of(a), 0x1p20f, 0x1p23f)) & 0x7Fu;
  return ((~ux >> 20) & 0x800u) | (a < 0x38800000u ? sub : mag_normal(a, carry));
}

/* general path, the value's own bits */
static uint32_t code_general(uint32_t u) {
  const uint32_t a = u & 0x7FFFFFFFu, sign12 = (u >> 20) & 0x800u;
  if (a > 0x7F800000u) return 0x7FFu;
  if (a >= 0x477E0000u) return sign12 | 0x7BFu;
  if (a < 0x38800000u) {
    /* an exact scaling by 2^20 (a power of two), then a round to nearest
     * even to an integer */
    return sign12 | (uint32_t)nearbyintf(f_of(a) * 0x1p20f);
  }
  const uint32_t r = (a + 0xFFFFu + ((a >> 17) & 1u)) & ~0x1FFFFu;
  return sign12 | (((r >> 23) - 112u) << 6) | ((r >> 17) & 0x3Fu);
}

/* decoder: codes 0..3 of a 48-bit group {hi16:lo} as four floats */
static void decode4(uint32_t lo, uint32_t hi16, float out[4]) {
  const uint32_t funnel = (uint32_t)((((uint64_t)hi16 << 32) | lo) >> 20);
  const uint32_t h01 = ((lo << 4) & 0x0000FFF0u) | ((lo << 8) & 0xFFF00000u);
  const uint32_t h23 = (funnel & 0x0000FFF0u) | ((hi16 << 16) & 0xFFF00000u);
  const uint32_t w[2] = {h01, h23};
  for (int i = 0; i < 4; ++i) {
    const uint16_t bits = (uint16_t)(w[i >> 1] >> (16 * (i & 1)));
    _Float16 h;
    memcpy(&h, &bits, 2);
    out[i] = (float)h;
  }
}

/* value of a code by its fields */
static double value_def(uint32_t c) {
  const double sign = (c & 0x800u) ? -1.0 : 1.0;
  const uint32_t e = (c >> 6) & 0x1Fu, m = c & 0x3Fu;
  if (e == 31) return m ? NAN : sign * INFINITY;
  if (e == 0) return sign * ldexp((double)m, -20);
  return sign * ldexp(1.0 + m / 64.0, (int)e - 15);
}

static void pack8(const uint32_t* c, uint32_t w[3]) {
  w[0] = c[0] | (c[1] << 12) | (c[2] << 24);
  w[1] = (c[2] >> 8) | (c[3] << 4) | (c[4] << 16) | (c[5] << 28);
  w[2] = (c[5] >> 4) | (c[6] << 8) | (c[7] << 20);
}

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint32_t next_code(void) { /* splitmix64, low 12 bits */
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return (uint32_t)(z ^ (z >> 31)) & 0xFFFu;
}

static long long pairs, mismatches;

static void check_fast(int carry) {
  long long n = 0, bad = 0;
  int printed = 0;
#pragma omp parallel for reduction(+ : n, bad) schedule(static)
  for (long long a = 0; a < 0x477F0000ll; ++a) {
    for (int s = 0; s < 2; ++s) {
      const uint32_t ux = (uint32_t)a | (s ? 0x80000000u : 0u);
      const uint32_t got = code_fast(ux, carry), want = code_def(-f_of(ux));
      ++n;
      if (got != want) {
        ++bad;
#pragma omp critical
        if (printed < 10) {
          printf("mismatch q=%a code=%03x want=%03x\n", f_of(ux), got, want);
          ++printed;
        }
      }
    }
  }
  pairs = n;
  mismatches = bad;
}

static void check_general(void) {
  long long n = 0, bad = 0;
  int printed = 0;
#pragma omp parallel for reduction(+ : n, bad) schedule(static)
  for (long long u = 0; u <= 0xFFFFFFFFll; ++u) {
    const uint32_t got = code_general((uint32_t)u), want = code_def(f_of((uint32_t)u));
    ++n;
    if (got != want) {
      ++bad;
#pragma omp critical
      if (printed < 10) {
        printf("mismatch y=%a code=%03x want=%03x\n", f_of((uint32_t)u), got, want);
        ++printed;
      }
    }
  }
  pairs = n;
  mismatches = bad;
}

static void check_decode(void) {
  int printed = 0;
  for (int pos = 0; pos < 4; ++pos) {
    for (int rep = 0; rep < 16; ++rep) {
      for (uint32_t c = 0; c < 4096; ++c) {
        uint32_t codes[4];
        for (int i = 0; i < 4; ++i) codes[i] = (i == pos) ? c : next_code();
        uint64_t v = 0;
        for (int i = 0; i < 4; ++i) v |= (uint64_t)codes[i] << (12 * i);
        float got[4];
        decode4((uint32_t)v, (uint32_t)(v >> 32), got);
        for (int i = 0; i < 4; ++i) {
          const double want = value_def(codes[i]);
          const int ok = isnan(want) ? isnan(got[i])
                                     : ((double)got[i] == want &&
                                        !signbit(got[i]) == !signbit(want));
          ++pairs;
          if (!ok) {
            ++mismatches;
            if (printed++ < 10) printf("mismatch code=%03x got=%a want=%a\n", codes[i], got[i], want);
          }
        }
      }
    }
  }
}

static void check_pack(long long n) {
  int printed = 0;
  for (long long t = 0; t < n; ++t) {
    uint32_t c[8], w[3];
    for (int i = 0; i < 8; ++i) c[i] = next_code();
    pack8(c, w);
    for (int i = 0; i < 8; ++i) {
      uint32_t got = 0;
      for (int b = 0; b < 12; ++b) {
        const int bit = 12 * i + b;
        got |= ((w[bit >> 5] >> (bit & 31)) & 1u) << b;
      }
      ++pairs;
      if (got != c[i]) {
        ++mismatches;
        if (printed++ < 10) printf("mismatch element %d code=%03x got=%03x\n", i, c[i], got);
      }
    }
  }
}

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  if (!strcmp(argv[1], "fast"))
    check_fast(1);
  else if (!strcmp(argv[1], "fast_nocarry"))
    check_fast(0);
  else if (!strcmp(argv[1], "general"))
    check_general();
  else if (!strcmp(argv[1], "decode"))
    check_decode();
  else if (!strcmp(argv[1], "pack") && argc >= 3)
    check_pack(atoll(argv[2]));
  else
    return 2;
  printf("pairs=%lld mismatches=%lld\n", pairs, mismatches);
  return 0;
}
