/*
 * fp8bs_oracle.c -- plain CPU oracle for fine-grained FP8 quantization and
 * the block-scaled FP8 GEMM.  TEST INFRASTRUCTURE ONLY (see the header).
 *
 * Everything here is written straight from the definitions: the E4M3 value
 * of a code, nearest-value rounding found by search over the 127 finite
 * non-negative codes, one correctly rounded FP32 division per scale and per
 * element, and double-precision dot products.  No blocking, vectorisation
 * tricks or shared tables with the CUDA library.  Build with -O2
 * -ffp-contract=off and never with -ffast-math: the FP32 divisions and
 * multiplies must be the IEEE round-to-nearest ones.
 */
#include "fp8bs_oracle.h"

#include <math.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define GROUP 128 /* [P1¶3] 1x128 tiles, 128x128 blocks */
#define E4M3_MAX 448.0 /* largest finite E4M3FN value: 1.75 * 2^8 (R1) */

/* ------------------------------------------------------------------------ */
/* E4M3 codec                                                                */
/* ------------------------------------------------------------------------ */

/* Code layout S EEEE MMM, exponent bias 7.  Exponent field 0 holds the
 * subnormals m * 2^-9; otherwise the value is (1 + m/8) * 2^(e-7), which is
 * (8 + m) * 2^(e-10).  S.1111.111 is NaN; there is no infinity (R1). */
double fp8bs_oracle_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return sign ? -v : v;
}

/* Nearest E4M3 value to y; ties go to the code whose mantissa LSB (the code
 * LSB) is 0.  Codes 0x00..0x7E are the non-negative finite values in
 * increasing order, so a binary search over code numbers finds the two
 * neighbours of |y|.  Finite |y| >= 448 and +-Inf saturate to 448 (R8);
 * NaN gives 0x7F. */
uint8_t fp8bs_oracle_e4m3_encode(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= E4M3_MAX) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E; /* decode(lo) <= a < decode(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (fp8bs_oracle_e4m3_decode((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  double below = a - fp8bs_oracle_e4m3_decode((uint8_t)lo);
  double above = fp8bs_oracle_e4m3_decode((uint8_t)hi) - a;
  int c;
  if (below < above)
    c = lo;
  else if (above < below)
    c = hi;
  else
    c = (lo & 1) ? hi : lo; /* exact tie: even mantissa */
  return (uint8_t)(sign | c);
}

float fp8bs_oracle_bf16_to_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* bf16 has 8 significant bits and the FP32 exponent range, so its spacing
 * around |v| in [2^e, 2^(e+1)) is 2^(e-7), and 2^-133 below 2^-126. */
uint16_t fp8bs_oracle_double_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): leading bit is 2^(e-1) */
  int ulp_exp = (e - 1) - 7;
  if (ulp_exp < -133) ulp_exp = -133;
  double r = nearbyint(ldexp(a, -ulp_exp)); /* default mode: ties to even */
  double rv = ldexp(r, ulp_exp);
  if (rv >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float f = (float)rv; /* exact: rv has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

/* ------------------------------------------------------------------------ */
/* One group: amax, scale, codes                                             */
/* ------------------------------------------------------------------------ */

/* |v| with NaN ignored (R5). */
static float amax_update(float amax, float v) {
  float a = fabsf(v);
  if (isnan(a)) return amax;
  return a > amax ? a : amax;
}

/* [P1¶3] "derive the scaling factor": s = amax / 448 (R2). */
static float scale_of(float amax) { return amax / (float)E4M3_MAX; }

/* [P1¶3] "quantize ... online into the FP8 format": code of x under s (R3,
 * R4, R5). */
static uint8_t code_of(float x, float s) {
  if (isnan(x)) return 0x7F;
  if (s == 0.0f) return signbit(x) ? 0x80 : 0x00;
  float y = x / s;
  return fp8bs_oracle_e4m3_encode(y);
}

/* ------------------------------------------------------------------------ */
/* Quantizers                                                                */
/* ------------------------------------------------------------------------ */

void fp8bs_oracle_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K,
                                  uint8_t *q, float *s) {
  int64_t KB = K / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t kb = 0; kb < KB; ++kb) {
      const uint16_t *row = x + m * K + kb * GROUP;
      float amax = 0.0f;
      for (int j = 0; j < GROUP; ++j)
        amax = amax_update(amax, fp8bs_oracle_bf16_to_float(row[j]));
      float sc = scale_of(amax);
      s[kb * M + m] = sc;
      for (int j = 0; j < GROUP; ++j)
        q[m * K + kb * GROUP + j] =
            code_of(fp8bs_oracle_bf16_to_float(row[j]), sc);
    }
  }
}

void fp8bs_oracle_quant_f32_1x128(const float *x, int64_t M, int64_t K,
                                  uint8_t *q, float *s) {
  int64_t KB = K / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t kb = 0; kb < KB; ++kb) {
      const float *row = x + m * K + kb * GROUP;
      float amax = 0.0f;
      for (int j = 0; j < GROUP; ++j) amax = amax_update(amax, row[j]);
      float sc = scale_of(amax);
      s[kb * M + m] = sc;
      for (int j = 0; j < GROUP; ++j) q[m * K + kb * GROUP + j] = code_of(row[j], sc);
    }
  }
}

void fp8bs_oracle_quant_per_tensor(const uint16_t *x, int64_t rows,
                                   int64_t cols, uint8_t *q, float *s) {
  int64_t n = rows * cols;
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i)
    amax = amax_update(amax, fp8bs_oracle_bf16_to_float(x[i]));
  float sc = scale_of(amax);
  *s = sc;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    q[i] = code_of(fp8bs_oracle_bf16_to_float(x[i]), sc);
}

void fp8bs_oracle_quant_act_128x1(const uint16_t *x, int64_t M, int64_t N,
                                  uint8_t *qT, float *sT) {
  /* Literally: transpose, then 1x128 tiles along the new rows. */
  int64_t MB = M / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t mb = 0; mb < MB; ++mb) {
      float amax = 0.0f;
      for (int j = 0; j < GROUP; ++j)
        amax = amax_update(
            amax, fp8bs_oracle_bf16_to_float(x[(mb * GROUP + j) * N + n]));
      float sc = scale_of(amax);
      sT[mb * N + n] = sc;
      for (int j = 0; j < GROUP; ++j)
        qT[n * M + mb * GROUP + j] = code_of(
            fp8bs_oracle_bf16_to_float(x[(mb * GROUP + j) * N + n]), sc);
    }
  }
}

void fp8bs_oracle_quant_weight_128x128(const uint16_t *w, int64_t N,
                                       int64_t K, uint8_t *q, float *s,
                                       uint8_t *qT, float *sT) {
  int64_t NB = N / GROUP, KB = K / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t blk = 0; blk < NB * KB; ++blk) {
    int64_t nb = blk / KB, kb = blk % KB;
    float amax = 0.0f;
    for (int i = 0; i < GROUP; ++i)
      for (int j = 0; j < GROUP; ++j)
        amax = amax_update(amax, fp8bs_oracle_bf16_to_float(
                                     w[(nb * GROUP + i) * K + kb * GROUP + j]));
    float sc = scale_of(amax);
    s[nb * KB + kb] = sc;
    if (sT) sT[kb * NB + nb] = sc;
    for (int i = 0; i < GROUP; ++i) {
      for (int j = 0; j < GROUP; ++j) {
        int64_t n = nb * GROUP + i, k = kb * GROUP + j;
        uint8_t c = code_of(fp8bs_oracle_bf16_to_float(w[n * K + k]), sc);
        q[n * K + k] = c;
        if (qT) qT[k * N + n] = c;
      }
    }
  }
}

/* R7: x_hat = fl32(decode(q) * s), then 128x1 groups of x_hat. */
static float dequant_one(const uint8_t *q, const float *s, int64_t M,
                         int64_t K, int64_t m, int64_t k) {
  float d = (float)fp8bs_oracle_e4m3_decode(q[m * K + k]);
  return d * s[(k / GROUP) * M + m];
}

void fp8bs_oracle_requant_1x128_to_128x1(const uint8_t *q, const float *s,
                                         int64_t M, int64_t K, uint8_t *qT,
                                         float *sT) {
  int64_t MB = M / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < K; ++k) {
    for (int64_t mb = 0; mb < MB; ++mb) {
      float amax = 0.0f;
      for (int j = 0; j < GROUP; ++j)
        amax = amax_update(amax, dequant_one(q, s, M, K, mb * GROUP + j, k));
      float sc = scale_of(amax);
      sT[mb * K + k] = sc;
      for (int j = 0; j < GROUP; ++j)
        qT[k * M + mb * GROUP + j] =
            code_of(dequant_one(q, s, M, K, mb * GROUP + j, k), sc);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* E5M6 (readings R9-R12)                                                    */
/* ------------------------------------------------------------------------ */

#define E5M6_MAX 65024.0 /* (1 + 63/64) * 2^15, code 0x7BF */

/* Layout S EEEEE MMMMMM, bias 15: (64 + m) * 2^(e-21) for e >= 1,
 * m * 2^-20 for e == 0. */
double fp8bs_oracle_e5m6_decode(uint16_t code) {
  int sign = (code >> 11) & 1;
  int e = (code >> 6) & 0x1F;
  int m = code & 0x3F;
  double v;
  if (e == 31)
    v = (m == 0) ? INFINITY : NAN;
  else
    v = (e == 0) ? ldexp((double)m, -20) : ldexp((double)(64 + m), e - 21);
  return sign ? -v : v;
}

/* Codes 0x000..0x7BF are the non-negative finite values in increasing order:
 * a binary search finds the neighbours of |y|, as for E4M3. */
uint16_t fp8bs_oracle_e5m6_encode(float y) {
  if (isnan(y)) return 0x7FF;
  uint16_t sign = signbit(y) ? 0x800 : 0x000;
  double a = fabs((double)y);
  if (a >= E5M6_MAX) return (uint16_t)(sign | 0x7BF);
  int lo = 0, hi = 0x7BF; /* decode(lo) <= a < decode(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (fp8bs_oracle_e5m6_decode((uint16_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  double below = a - fp8bs_oracle_e5m6_decode((uint16_t)lo);
  double above = fp8bs_oracle_e5m6_decode((uint16_t)hi) - a;
  int c;
  if (below < above)
    c = lo;
  else if (above < below)
    c = hi;
  else
    c = (lo & 1) ? hi : lo;
  return (uint16_t)(sign | c);
}

void fp8bs_oracle_e5m6_pack(const uint16_t *codes, int64_t n, uint8_t *packed) {
  for (int64_t i = 0; i < n; i += 2) {
    uint32_t c0 = codes[i] & 0xFFF, c1 = codes[i + 1] & 0xFFF;
    uint32_t bitsv = c0 | (c1 << 12); /* bits 12i .. 12i+23 of the stream */
    packed[3 * (i / 2)] = (uint8_t)(bitsv & 0xFF);
    packed[3 * (i / 2) + 1] = (uint8_t)((bitsv >> 8) & 0xFF);
    packed[3 * (i / 2) + 2] = (uint8_t)((bitsv >> 16) & 0xFF);
  }
}

void fp8bs_oracle_e5m6_unpack(const uint8_t *packed, int64_t n,
                              uint16_t *codes) {
  for (int64_t i = 0; i < n; i += 2) {
    uint32_t bitsv = (uint32_t)packed[3 * (i / 2)] |
                     ((uint32_t)packed[3 * (i / 2) + 1] << 8) |
                     ((uint32_t)packed[3 * (i / 2) + 2] << 16);
    codes[i] = (uint16_t)(bitsv & 0xFFF);
    codes[i + 1] = (uint16_t)(bitsv >> 12);
  }
}

/* R10: scale and code of one element under the E5M6 maximum. */
static float scale_of_e5m6(float amax) { return amax / (float)E5M6_MAX; }

static uint16_t code_of_e5m6(float x, float s) {
  if (isnan(x)) return 0x7FF;
  if (s == 0.0f) return signbit(x) ? 0x800 : 0x000;
  return fp8bs_oracle_e5m6_encode(x / s);
}

void fp8bs_oracle_quant_act_e5m6_1x128(const uint16_t *x, int64_t M,
                                       int64_t K, uint8_t *packed, float *s) {
  int64_t KB = K / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    uint16_t codes[GROUP];
    for (int64_t kb = 0; kb < KB; ++kb) {
      const uint16_t *row = x + m * K + kb * GROUP;
      float amax = 0.0f;
      for (int j = 0; j < GROUP; ++j)
        amax = amax_update(amax, fp8bs_oracle_bf16_to_float(row[j]));
      float sc = scale_of_e5m6(amax);
      s[kb * M + m] = sc;
      for (int j = 0; j < GROUP; ++j)
        codes[j] = code_of_e5m6(fp8bs_oracle_bf16_to_float(row[j]), sc);
      /* a 128-element group starts on a whole byte: bit 12 * 128 * kb */
      fp8bs_oracle_e5m6_pack(codes, GROUP,
                             packed + m * (K / 2 * 3) + kb * (GROUP / 2 * 3));
    }
  }
}

void fp8bs_oracle_requant_e5m6_to_128x1(const uint8_t *packed, const float *s,
                                        int64_t M, int64_t K, uint8_t *qT,
                                        float *sT) {
  int64_t MB = M / GROUP, KB = K / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t kb = 0; kb < KB; ++kb) {
    float xh[GROUP][GROUP]; /* [row within the block][column] */
    uint16_t codes[GROUP];
    for (int64_t mb = 0; mb < MB; ++mb) {
      for (int j = 0; j < GROUP; ++j) {
        int64_t m = mb * GROUP + j;
        fp8bs_oracle_e5m6_unpack(packed + m * (K / 2 * 3) + kb * (GROUP / 2 * 3),
                                 GROUP, codes);
        for (int c = 0; c < GROUP; ++c)
          xh[j][c] = (float)fp8bs_oracle_e5m6_decode(codes[c]) * s[kb * M + m];
      }
      for (int c = 0; c < GROUP; ++c) {
        int64_t k = kb * GROUP + c;
        float amax = 0.0f;
        for (int j = 0; j < GROUP; ++j) amax = amax_update(amax, xh[j][c]);
        float sc = scale_of(amax);
        sT[mb * K + k] = sc;
        for (int j = 0; j < GROUP; ++j)
          qT[k * M + mb * GROUP + j] = code_of(xh[j][c], sc);
      }
    }
  }
}

void fp8bs_oracle_quant_rowwise(const uint16_t *x, int64_t M, int64_t K,
                                uint8_t *q, float *s) {
  int64_t KB = K / GROUP;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k)
      amax = amax_update(amax, fp8bs_oracle_bf16_to_float(x[m * K + k]));
    float sc = scale_of(amax);
    for (int64_t kb = 0; kb < KB; ++kb) s[kb * M + m] = sc;
    for (int64_t k = 0; k < K; ++k)
      q[m * K + k] = code_of(fp8bs_oracle_bf16_to_float(x[m * K + k]), sc);
  }
}

/* ------------------------------------------------------------------------ */
/* GEMM                                                                      */
/* ------------------------------------------------------------------------ */

/* Scale of B's element (n, k): one per 128x128 block, or one per 1x128 tile
 * of row n (the weight-gradient GEMM, whose B operand is an activation). */
static double b_scale(const float *sb, int bkind, int64_t N, int64_t K,
                      int64_t n, int64_t k) {
  if (bkind == FP8BS_ORACLE_BSCALE_BLOCK_128x128)
    return (double)sb[(n / GROUP) * (K / GROUP) + k / GROUP];
  return (double)sb[(k / GROUP) * N + n];
}

/* [P1¶2] each K-group's contribution carries its own scale pair; with exact
 * arithmetic the promotion schedule disappears and C is just the sum of the
 * dequantized products. */
static double dot_dequant(const uint8_t *a, const float *sa, const uint8_t *b,
                          const float *sb, int bkind, int64_t M, int64_t N,
                          int64_t K, int64_t m, int64_t n) {
  double acc = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double av = fp8bs_oracle_e4m3_decode(a[m * K + k]) *
                (double)sa[(k / GROUP) * M + m];
    double bv = fp8bs_oracle_e4m3_decode(b[n * K + k]) *
                b_scale(sb, bkind, N, K, n, k);
    acc += av * bv;
  }
  return acc;
}

void fp8bs_oracle_gemm(const uint8_t *a, const float *sa, const uint8_t *b,
                       const float *sb, int bkind, int64_t M, int64_t N,
                       int64_t K, double *c) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      c[m * N + n] = dot_dequant(a, sa, b, sb, bkind, M, N, K, m, n);
}

void fp8bs_oracle_gemm_sampled(const uint8_t *a, const float *sa,
                               const uint8_t *b, const float *sb, int bkind,
                               int64_t M, int64_t N, int64_t K,
                               const int64_t *ms, const int64_t *ns,
                               int64_t count, double *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i)
    out[i] = dot_dequant(a, sa, b, sb, bkind, M, N, K, ms[i], ns[i]);
}

/* ------------------------------------------------------------------------ */
/* Limited-precision accumulator model (PARITY UNPINNED)                     */
/* ------------------------------------------------------------------------ */

/* floor(log2|v|) for v != 0. */
static int exponent_of(double v) {
  int e;
  frexp(v, &e);
  return e - 1;
}

/* Truncate toward zero to a 24-bit significand (FP32 without rounding up). */
static double trunc_to_fp32(double v) {
  if (v == 0.0) return 0.0;
  int e = exponent_of(fabs(v));
  int ulp = e - 23;
  if (ulp < -149) ulp = -149;
  return ldexp(trunc(ldexp(v, -ulp)), ulp);
}

void fp8bs_oracle_gemm_limited_acc(const uint8_t *a, const float *sa,
                                   const uint8_t *b, const float *sb,
                                   int bkind, int64_t M, int64_t N, int64_t K,
                                   int bits, int group, int promote_every,
                                   const int64_t *ms, const int64_t *ns,
                                   int64_t count, double *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    int64_t m = ms[i], n = ns[i];
    double acc = 0.0;   /* the modelled tensor-core accumulator */
    double total = 0.0; /* the promoted sum, kept in double */
    for (int64_t k0 = 0; k0 < K; k0 += group) {
      /* [P2¶3] align the group's products and the running sum to the
       * largest exponent, keep `bits` bits below it (sign-fill right shift
       * = floor on the two's-complement value), add exactly. */
      int have = acc != 0.0;
      int emax = have ? exponent_of(fabs(acc)) : 0;
      for (int j = 0; j < group && k0 + j < K; ++j) {
        double p = fp8bs_oracle_e4m3_decode(a[m * K + k0 + j]) *
                   fp8bs_oracle_e4m3_decode(b[n * K + k0 + j]);
        if (p != 0.0) {
          int e = exponent_of(fabs(p));
          if (!have || e > emax) emax = e;
          have = 1;
        }
      }
      if (have) {
        double unit = ldexp(1.0, emax - bits + 1);
        double sum = floor(acc / unit);
        for (int j = 0; j < group && k0 + j < K; ++j) {
          double p = fp8bs_oracle_e4m3_decode(a[m * K + k0 + j]) *
                     fp8bs_oracle_e4m3_decode(b[n * K + k0 + j]);
          sum += floor(p / unit);
        }
        acc = trunc_to_fp32(sum * unit);
      }
      int64_t done = k0 + group;
      if (promote_every > 0 && (done % promote_every == 0 || done >= K)) {
        int64_t kb = k0 / GROUP;
        total += acc * (double)sa[kb * M + m] *
                 b_scale(sb, bkind, N, K, n, kb * GROUP);
        acc = 0.0;
      }
    }
    if (promote_every > 0)
      out[i] = total;
    else
      out[i] = acc * (double)sa[m] * b_scale(sb, bkind, N, K, n, 0);
  }
}

int fp8bs_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
