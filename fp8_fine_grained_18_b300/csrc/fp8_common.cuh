// fp8_common.cuh -- device helpers shared by the libfp8bs kernels:
// bf16 unpacking, E4M3 packing/unpacking through the hardware converters,
// and the per-group scale and quotient arithmetic of the quantizers.
//
// Quantization rule (one group = a 1x128 tile, a 128x1 tile or a 128x128
// block; DeepSeek-V3 fine-grained quantization, page P1 paragraph 3):
//   amax = max |x| over the group (NaN ignored, Inf included)
//   s    = fl32(amax / 448)                      (one IEEE division)
//   code = E4M3_RNE_satfinite(fl32(x / s))       (two roundings)
//   s == 0      -> every non-NaN element codes as a zero of its own sign
//   NaN element -> 0x7F
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace fp8bs {

constexpr int kGroup = 128;          // 1x128 tiles, 128x128 blocks
constexpr float kE4M3Max = 448.0f;   // largest finite E4M3FN value
constexpr float kE5M6Max = 65024.0f;  // largest finite E5M6 value (1.984375 * 2^15)
// Below this scale the reciprocal-based quotient can meet FP32 subnormals;
// such groups take the exact-division path.
constexpr float kFastScaleMin = 0x1.0p-92f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> two E4M3 codes (RNE, saturate to +-448); lo in byte 0.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (byte 0 = first) -> two exact floats.
__device__ __forceinline__ float2 e4m3x2_decode(uint32_t two_codes) {
  uint32_t h2;
  uint16_t in = (uint16_t)two_codes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  float lo, hi;
  asm("{.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;}"
      : "=f"(lo), "=f"(hi) : "r"(h2));
  return make_float2(lo, hi);
}

// Scale of a group whose max magnitude is amax, for a format whose largest
// finite value is fmt_max (448 for E4M3; 65024 for the E5M6 cache).
__device__ __forceinline__ float group_scale(float amax, float fmt_max = kE4M3Max) {
  return __fdiv_rn(amax, fmt_max);
}

// Fast path: a normal, finite scale s with nr = -fl32(1/s) (a correctly
// rounded reciprocal, negated).  The quotient is formed negated, by one
// Markstein correction step (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", 1990) with every
// operation rounded once:
//   Q0 = x * nr,  e = fma(Q0, s, x) (= x - s * q0, exact),  Q = fma(e, nr, Q0)
// which is -fl32(x / s): round-to-nearest is symmetric under negation, and
// in this arrangement a zero quotient also comes out with the opposite of
// x's sign, so -Q carries x's sign in every case.  The caller converts Q to
// E4M3 and flips the sign bit of each code.  For the bf16 inputs of the
// activation and weight quantizers one step reproduces fl32(x/s) wherever
// |x/s| >= 2^-12 (checked exhaustively over bf16 inputs against IEEE
// division); below that every candidate codes as a zero of x's sign.
// Two packed FP32 lanes are processed per instruction.
__device__ __forceinline__ float2 neg_quotient_1step_x2(float2 x, float s, float nr) {
  const float2 nr2 = make_float2(nr, nr), s2 = make_float2(s, s);
  const float2 q0 = ptx::mul2_rn(x, nr2);
  const float2 e = ptx::fma2_rn(q0, s2, x);
  return ptx::fma2_rn(e, nr2, q0);
}

// Two correction steps: the first makes the quotient faithful for any FP32
// x, the second then yields the correctly rounded quotient (Markstein's
// theorem).  Used where x is a full 24-bit FP32 value (the requantizer).
__device__ __forceinline__ float2 neg_quotient_2step_x2(float2 x, float s, float nr) {
  const float2 nr2 = make_float2(nr, nr), s2 = make_float2(s, s);
  const float2 q0 = ptx::mul2_rn(x, nr2);
  const float2 e0 = ptx::fma2_rn(q0, s2, x);
  const float2 q1 = ptx::fma2_rn(e0, nr2, q0);
  const float2 e1 = ptx::fma2_rn(q1, s2, x);
  return ptx::fma2_rn(e1, nr2, q1);
}

// General path for one element: exact division and every special case.
__device__ __forceinline__ float quotient_general(float x, float s) {
  if (x != x) return x;  // NaN stays NaN
  if (s == 0.0f) return __uint_as_float(__float_as_uint(x) & 0x80000000u);
  return __fdiv_rn(x, s);
}

// Codes of two quotients with NaN -> 0x7F made explicit.
__device__ __forceinline__ uint32_t e4m3x2_nan(float lo, float hi) {
  uint32_t c = e4m3x2(lo, hi);
  if (lo != lo) c = (c & 0xFF00u) | 0x7Fu;
  if (hi != hi) c = (c & 0x00FFu) | 0x7F00u;
  return c;
}

// Max of |x| that propagates NaN (a NaN in the group shows up as NaN).
__device__ __forceinline__ float fmax_abs_nan(float acc, float x) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(acc), "f"(fabsf(x)));
  return r;
}

struct GroupScale {
  float s, nr;  // scale, and -fl32(1 / s) on the fast path
  bool fast;
};

// Scale of a group from its amax given as a bit pattern (bf16 when bf16 is
// true, else FP32); special = the group holds Inf or NaN.
__device__ __forceinline__ GroupScale make_scale(uint32_t mag_no_nan_bits, bool special,
                                                 bool bf16, float fmt_max = kE4M3Max) {
  GroupScale g;
  g.s = group_scale(__uint_as_float(bf16 ? mag_no_nan_bits << 16 : mag_no_nan_bits), fmt_max);
  g.fast = !special && g.s >= kFastScaleMin;
  g.nr = g.fast ? -__frcp_rn(g.s) : 0.0f;
  return g;
}

// Four FP32 values (full 24-bit significands) -> four codes.
__device__ __forceinline__ uint32_t codes_f32x4(float a, float b, float c, float d,
                                                const GroupScale& g) {
  if (g.fast) {
    const float2 q0 = neg_quotient_2step_x2(make_float2(a, b), g.s, g.nr);
    const float2 q1 = neg_quotient_2step_x2(make_float2(c, d), g.s, g.nr);
    return (e4m3x2(q0.x, q0.y) | (e4m3x2(q1.x, q1.y) << 16)) ^ 0x80808080u;
  }
  return e4m3x2_nan(quotient_general(a, g.s), quotient_general(b, g.s)) |
         (e4m3x2_nan(quotient_general(c, g.s), quotient_general(d, g.s)) << 16);
}

// ---------------------------------------------------------------------------
// E5M6, the 12-bit cache format of the activations that are re-tiled from
// 1x128 to 128x1 tiles (page P1, paragraph 3): sign, 5 exponent bits (bias
// 15), 6 mantissa bits; exponent 0 holds the subnormals m * 2^-20, exponent
// 31 Inf/NaN.  Rounding to nearest even, saturating at 65024; NaN -> 0x7FF.
// Codes are stored as a little-endian 12-bit stream (element i at bits
// 12i .. 12i+11 of its row).
// ---------------------------------------------------------------------------

// Code of the FP32 value with magnitude bits `a` (no sign bit) and sign
// `sign12` (0 or 0x800).
__device__ __forceinline__ uint32_t e5m6_code(uint32_t a, uint32_t sign12) {
  if (a > 0x7F800000u) return 0x7FFu;                      // NaN
  if (a >= 0x477E0000u) return sign12 | 0x7BFu;            // >= 65024 (and Inf): saturate
  if (a < 0x38800000u)                                     // below 2^-14: subnormal
    return sign12 | __float2uint_rn(__uint_as_float(a) * 0x1.0p20f);  // exact scaling; 64 = 2^-14
  // normal: round the FP32 significand to 6 bits, ties to even; a carry
  // moves into the exponent field, and nothing below 65024 rounds past it
  const uint32_t r = (a + 0xFFFFu + ((a >> 17) & 1u)) & ~0x1FFFFu;
  return sign12 | (((r >> 23) - 112u) << 6) | ((r >> 17) & 0x3Fu);
}

// Code of y (any FP32 value, the exact-division path).
__device__ __forceinline__ uint32_t e5m6_of(float y) {
  const uint32_t u = __float_as_uint(y);
  return e5m6_code(u & 0x7FFFFFFFu, (u >> 20) & 0x800u);
}

// Eight codes -> the 96-bit little-endian stream, as three words.
__device__ __forceinline__ uint3 e5m6_pack8(const uint32_t* c) {
  return make_uint3(c[0] | (c[1] << 12) | (c[2] << 24),
                    (c[2] >> 8) | (c[3] << 4) | (c[4] << 16) | (c[5] << 28),
                    (c[5] >> 4) | (c[6] << 8) | (c[7] << 20));
}

}  // namespace fp8bs
