/*
 * fp8bs_oracle.h -- plain, slow, obviously-correct CPU oracle for the
 * fine-grained FP8 quantizers and the block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library (libfp8bs); the two are
 * compared against each other, never built from each other.
 *
 * Citations name the five scraped pages that quote the DeepSeek-V3 technical
 * report as P1..P5 (page order as delivered) and their paragraphs as ¶1..¶5:
 *   P1 = xn--9g3bo1gtkw0l8ubf92bgle.kr qna wr_id=32373  (fine-grained
 *        quantization, online max-abs, 1x128 / 128x128 tiles, 14-bit
 *        accumulation, K=4096 ~2% error)
 *   P2 = why-be.why-be.co.kr as_center wr_id=73620       (accumulator
 *        mechanism "highest 14 bits ... sign-fill right shift ... truncate";
 *        HBM round trip of quantization)
 *   P3 = xn--9g3bo1gtkw0l8ubf92bgle.kr qna wr_id=113503  (per-tensor scaling
 *        is outlier-sensitive; backward for input / for weights)
 *   P4 = bestpmk.kr free wr_id=299512                    (FP8 GEMMs take FP8
 *        inputs and produce BF16 or FP32 outputs)
 *   P5 = blog.cameseeing.com freeboard wr_id=1551483     (no hot-path content)
 *
 * Readings where the pages are silent (each one is a choice, stated once):
 *   R1  FP8 format is OCP E4M3FN (bias 7, no Inf, NaN = S.1111.111, max 448).
 *   R2  scale s = fl32(amax / 448) by one correctly rounded division; no
 *       epsilon floor; scales stored as FP32.
 *   R3  code = E4M3_RNE_satfinite(fl32(x / s)): two roundings, on purpose.
 *   R4  all-zero group (amax == 0): s = 0, non-NaN elements encode as zero
 *       with their own sign; 0/0 is never evaluated.
 *   R5  amax ignores NaN and includes Inf; a NaN element always encodes as
 *       0x7F; an Inf in a group makes s = Inf, so finite elements become
 *       signed zero and the Inf element becomes NaN (Inf/Inf).
 *   R6  IEEE subnormals everywhere (no flush to zero).
 *   R7  the requantizer starts from the cached FP8 codes and their scales,
 *       dequantizing with one round-to-nearest FP32 multiply.
 *   R8  the encoder saturates every finite |y| > 448 and every infinity to
 *       448 with y's sign (satfinite).
 *
 * Scale layouts (all FP32, row-major):
 *   1x128 groups of an operand X[rows][cols]:  s[cols/128][rows]
 *   128x128 blocks of W[N][K]:                 s[N/128][K/128]
 *   the transposed weight copy W^T[K][N]:      sT[K/128][N/128]
 */
#ifndef FP8BS_ORACLE_H
#define FP8BS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* --- E4M3 codec (OCP FP8 E4M3FN definition; reading R1, R8) ------------ */

/* Value of an E4M3 code, in double (exact).  NaN codes return NaN. */
double fp8bs_oracle_e4m3_decode(uint8_t code);

/* Round-to-nearest-even with saturation of a float to E4M3. */
uint8_t fp8bs_oracle_e4m3_encode(float y);

/* Value of a bf16 bit pattern, as float (exact). */
float fp8bs_oracle_bf16_to_float(uint16_t bits);

/* Round a double to the nearest bf16 (ties to even); returns the bits. */
uint16_t fp8bs_oracle_double_to_bf16(double v);

/* --- Quantizers ---------------------------------------------------------- */

/* [P1¶3] one scale per 1x128 activation tile, from the tile's online amax.
 * x: bf16 bits [M][K], K % 128 == 0.  q: [M][K].  s: [K/128][M]. */
void fp8bs_oracle_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K,
                                  uint8_t *q, float *s);

/* [P1¶3] the 1x128 rule applied to FP32 values (the output of a GEMM that is
 * quantized for the next layer): x: float [M][K], K % 128 == 0.
 * q: [M][K].  s: [K/128][M]. */
void fp8bs_oracle_quant_f32_1x128(const float *x, int64_t M, int64_t K,
                                  uint8_t *q, float *s);

/* [P1¶4][P3¶4] the standard practice the fine-grained tiles replace: one
 * scale for the whole tensor, its max-abs mapped to the FP8 maximum (the
 * accuracy baseline).  x: bf16 bits [rows][cols]; q: [rows][cols];
 * *s: the one scale (readings R2-R5 with a single group). */
void fp8bs_oracle_quant_per_tensor(const uint16_t *x, int64_t rows,
                                   int64_t cols, uint8_t *q, float *s);

/* [P1¶3] the same tiles laid along the other axis (128x1): groups are 128
 * consecutive rows of one column.  Equals quant_act_1x128 applied to the
 * transpose of x.  x: bf16 bits [M][N], M % 128 == 0.
 * qT: [N][M].  sT: [M/128][N]. */
void fp8bs_oracle_quant_act_128x1(const uint16_t *x, int64_t M, int64_t N,
                                  uint8_t *qT, float *sT);

/* [P1¶3] one scale per 128x128 weight block.  w: bf16 bits [N][K], N and K
 * multiples of 128.  q: [N][K]; s: [N/128][K/128].  qT (nullable): [K][N],
 * the same codes transposed; sT (nullable): [K/128][N/128]. */
void fp8bs_oracle_quant_weight_128x128(const uint16_t *w, int64_t N,
                                       int64_t K, uint8_t *q, float *s,
                                       uint8_t *qT, float *sT);

/* [P1¶3] 1x128 -> 128x1 transform for the backward pass (reading R7).
 * q: [M][K] codes with s: [K/128][M].  Output qT: [K][M], sT: [M/128][K].
 * M and K multiples of 128. */
void fp8bs_oracle_requant_1x128_to_128x1(const uint8_t *q, const float *s,
                                         int64_t M, int64_t K, uint8_t *qT,
                                         float *sT);

/* --- E5M6 cache of the re-tiled activations ([P1¶3]: the activations that
 * go from 1x128 to 128x1 tiles in the backward pass are kept in a custom
 * E5M6 format).  Readings:
 *   R9   E5M6 = sign, 5 exponent bits (bias 15), 6 mantissa bits.  Exponent
 *        field 0 holds the subnormals m * 2^-20; field 31 is Inf (m == 0)
 *        or NaN; the largest finite value is 1.984375 * 2^15 = 65024
 *        (code 0x7BF).  Rounding is to nearest, ties to even, saturating
 *        like R8; NaN encodes as 0x7FF.
 *   R10  the cache keeps the 1x128 tiles: s = fl32(amax / 65024) and
 *        code = E5M6(fl32(x / s)), R2-R6 with 65024 in place of 448.
 *   R11  codes are stored as a little-endian 12-bit stream: element i of a
 *        row occupies bits 12i .. 12i+11 of the row's 3K/2 bytes.
 *   R12  the backward re-tiling decodes x^ = fl32(decode(code) * s) (one
 *        rounding, as R7) and applies the 128x1 E4M3 rule to x^. */

/* Value of a 12-bit E5M6 code, in double (exact); NaN codes give NaN. */
double fp8bs_oracle_e5m6_decode(uint16_t code);

/* Nearest E5M6 code to y (R9). */
uint16_t fp8bs_oracle_e5m6_encode(float y);

/* n codes (n even) <-> 3n/2 bytes (R11). */
void fp8bs_oracle_e5m6_pack(const uint16_t *codes, int64_t n, uint8_t *packed);
void fp8bs_oracle_e5m6_unpack(const uint8_t *packed, int64_t n,
                              uint16_t *codes);

/* [P1¶3] x: bf16 [M][K] (K % 128 == 0) -> packed E5M6 [M][3K/2] bytes and
 * s: [K/128][M] (R10, R11). */
void fp8bs_oracle_quant_act_e5m6_1x128(const uint16_t *x, int64_t M,
                                       int64_t K, uint8_t *packed, float *s);

/* [P1¶3] the E5M6 cache re-tiled for the weight gradient: packed [M][3K/2],
 * s [K/128][M] -> qT: E4M3 [K][M], sT: [M/128][K] (R12); M % 128 == 0. */
void fp8bs_oracle_requant_e5m6_to_128x1(const uint8_t *packed, const float *s,
                                        int64_t M, int64_t K, uint8_t *qT,
                                        float *sT);

/* Test-only row-wise quantization (one group = a whole row of K); the
 * per-tensor/standard practice contrast of [P1¶4][P3¶4] applied per row.
 * Writes the row scale to every K-group slot: s: [K/128][M]. */
void fp8bs_oracle_quant_rowwise(const uint16_t *x, int64_t M, int64_t K,
                                uint8_t *q, float *s);

/* --- GEMM ------------------------------------------------------------------ */

#define FP8BS_ORACLE_BSCALE_BLOCK_128x128 0
#define FP8BS_ORACLE_BSCALE_TILE_1x128 1

/* [P1¶2][P4¶4] C[m][n] = sum_k (dec(a[m][k]) * sa(m,k)) * (dec(b[n][k]) *
 * sb(n,k)), summed in double.  a: [M][K], sa: [K/128][M]; b: [N][K];
 * sb: [N/128][K/128] (BLOCK) or [K/128][N] (TILE).  c: [M][N] double. */
void fp8bs_oracle_gemm(const uint8_t *a, const float *sa, const uint8_t *b,
                       const float *sb, int bkind, int64_t M, int64_t N,
                       int64_t K, double *c);

/* The same definition for a list of (m, n) output positions. */
void fp8bs_oracle_gemm_sampled(const uint8_t *a, const float *sa,
                               const uint8_t *b, const float *sb, int bkind,
                               int64_t M, int64_t N, int64_t K,
                               const int64_t *ms, const int64_t *ns,
                               int64_t count, double *out);

/* [P2¶3][P1¶3] PARITY UNPINNED (model, not a definition): a tensor-core
 * accumulator that keeps only the top `bits` bits of the aligned mantissas.
 * Every group of `group` products and the running sum are aligned to the
 * largest exponent among them, each truncated (two's-complement, toward
 * -inf) to a multiple of 2^(E-bits+1), summed exactly and truncated toward
 * zero back to FP32.  With promote_every > 0 the accumulator, times its
 * K-group's scales, is added into a double-precision sum every
 * promote_every products and reset (the model keeps the promoted side
 * exact, so only the limited accumulator loses precision); with
 * promote_every == 0 the whole K is
 * accumulated this way and the scales of K-group 0 are applied once at the
 * end (row-wise codes).  Computes a list of (m, n) outputs. */
void fp8bs_oracle_gemm_limited_acc(const uint8_t *a, const float *sa,
                                   const uint8_t *b, const float *sb,
                                   int bkind, int64_t M, int64_t N, int64_t K,
                                   int bits, int group, int promote_every,
                                   const int64_t *ms, const int64_t *ns,
                                   int64_t count, double *out);

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int fp8bs_oracle_num_threads(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_ORACLE_H */
