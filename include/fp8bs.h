/*
 * fp8bs.h -- C ABI of libfp8bs: fine-grained FP8 quantization and the
 * block-scaled FP8 GEMM that consumes it, for NVIDIA B300 (sm_103a).
 *
 * The method (DeepSeek-V3 FP8 training, as quoted by the five scraped pages
 * cited below as P1..P5 with their paragraphs as ¶n):
 *   - activations get one FP32 scale per 1x128 tile and weights one per
 *     128x128 block, each derived online from the tile's maximum absolute
 *     value, then cast to FP8 [P1¶3];
 *   - the scales run along the inner dimension K and are multiplied in on
 *     the CUDA cores while dequantizing [P1¶2], with partial sums promoted
 *     into FP32 because tensor-core accumulation alone is limited to about
 *     14 bits [P1¶3][P1¶4][P2¶3];
 *   - cached activations are re-tiled from 1x128 to 128x1 for the backward
 *     pass [P1¶3];
 *   - the GEMMs take FP8 inputs and write BF16 or FP32 [P4¶4];
 *   - the activations that are re-tiled are kept in a custom E5M6 format
 *     [P1¶3] (fp8bs_quant_act_e5m6, fp8bs_requant_e5m6_to_128x1);
 *   - one scale per tensor is the standard practice that the tiles replace,
 *     sensitive to outliers [P1¶4][P3¶4] (fp8bs_quant_per_tensor, kept as
 *     the accuracy baseline);
 *   - quantizing in a separate pass costs an HBM round trip [P2¶1]: the
 *     fused calls (fp8bs_quant_act_and_weight, fp8bs_quant_act_dual,
 *     fp8bs_gemm_quant_out) make several outputs from one read.
 * Page key: P1 = xn--9g3bo1gtkw0l8ubf92bgle.kr qna wr_id=32373,
 * P2 = why-be.why-be.co.kr as_center wr_id=73620,
 * P3 = xn--9g3bo1gtkw0l8ubf92bgle.kr qna wr_id=113503,
 * P4 = bestpmk.kr free wr_id=299512.
 *
 * Readings where the pages are silent: FP8 = OCP E4M3FN (max 448, NaN
 * 0x7F/0xFF, no infinity); scale s = fl32(amax / 448); code =
 * E4M3_round_nearest_even_satfinite(fl32(x / s)); amax ignores NaN and
 * includes Inf; an all-zero tile has s = 0 and signed-zero codes; a NaN
 * element codes as 0x7F; promotion happens once per 128-wide K group.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers, 16-byte aligned, dense row-major,
 *     owned and allocated by the caller, and must stay valid until the work
 *     queued on `stream` finishes.  The library allocates no per-call
 *     memory; outputs must not alias inputs.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and may be issued from several host threads on
 *     different streams.
 *   - Argument errors are detected on the host before anything is launched
 *     and returned synchronously; no output is touched in that case.
 *   - FP8BS_ERR_CUDA reports a failed CUDA call (the cudaError_t value is
 *     kept per host thread, see fp8bs_last_cuda_error()).
 *   - Scale layout for 1x128 groups of an operand X[rows][cols]:
 *     s[cols/128][rows] (FP32, rows contiguous).  Weight blocks of W[N][K]:
 *     s[N/128][K/128].
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, without requiring the CUDA headers. */
typedef struct CUstream_st *fp8bs_stream_t;

typedef enum {
  FP8BS_OK = 0,
  FP8BS_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum */
  FP8BS_ERR_UNSUPPORTED_SHAPE = 2, /* a size that is not a required multiple */
  FP8BS_ERR_MISALIGNED = 3,        /* a pointer not 16-byte aligned */
  FP8BS_ERR_ARCH = 4,              /* current device is not sm_103 */
  FP8BS_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed */
  FP8BS_ERR_TIMEOUT = 6            /* a bounded device wait gave up */
} fp8bs_status;

/* E4M3_1x128 is only for fp8bs_gemm_quant_out (it needs a scale array). */
typedef enum {
  FP8BS_OUT_BF16 = 0,
  FP8BS_OUT_F32 = 1,
  FP8BS_OUT_E4M3_1x128 = 2
} fp8bs_out_dtype;

typedef enum {
  /* B scales per 128x128 block: sb[N/128][K/128] (forward, input-grad) */
  FP8BS_BSCALE_BLOCK_128x128 = 0,
  /* B scales per 1x128 tile of each B row: sb[K/128][N] (weight-grad, whose
   * B operand is an activation re-tiled along tokens) */
  FP8BS_BSCALE_TILE_1x128 = 1
} fp8bs_bscale_kind;

/*
 * Activation quantizer [P1¶3]: one scale per 1x128 tile, from the tile's
 * online max-abs value.
 *
 * transpose_out == 0:
 *   x: bf16 [M][K] -> q: E4M3 [M][K], scales: f32 [K/128][M].
 *   Requires K % 128 == 0; M >= 0 (any M, including a ragged tail).
 * transpose_out == 1 (128x1 tiles for the weight-gradient GEMM, [P1¶3]):
 *   x: bf16 [M][K] -> q: E4M3 [K][M] (x transposed), scales: f32 [M/128][K]:
 *   the result equals mode 0 applied to the transpose of x.
 *   Requires M % 128 == 0 and K % 128 == 0.
 * M == 0 or K == 0 is a no-op returning FP8BS_OK.
 */
fp8bs_status fp8bs_quant_act_1x128(const void *x_bf16, int64_t M, int64_t K,
                                   int transpose_out, uint8_t *q,
                                   float *scales, fp8bs_stream_t stream);

/*
 * Both activation tilings of one tensor from a single read [P1¶3]: the
 * 1x128 tiles of fp8bs_quant_act_1x128(transpose_out = 0) and the 128x1
 * tiles of fp8bs_quant_act_1x128(transpose_out = 1), bit-identical to those
 * two calls.  Meant for grad_out, which feeds the input-gradient GEMM as
 * 1x128 tiles and the weight-gradient GEMM as 128x1 tiles; it reads the bf16
 * input from HBM once instead of twice.
 *   x: bf16 [M][K] -> q: E4M3 [M][K], scales: f32 [K/128][M]
 *                  -> qT: E4M3 [K][M], scalesT: f32 [M/128][K].
 *   Requires M % 128 == 0 and K % 128 == 0.
 */
fp8bs_status fp8bs_quant_act_dual(const void *x_bf16, int64_t M, int64_t K,
                                  uint8_t *q, float *scales, uint8_t *qT,
                                  float *scalesT, fp8bs_stream_t stream);

/*
 * Weight quantizer [P1¶3]: one scale per 128x128 block of W.
 *   w: bf16 [N][K] -> q: E4M3 [N][K], scales: f32 [N/128][K/128].
 *   qT (nullable): E4M3 [K][N], the same codes transposed (the K-major B
 *   operand of the input-gradient GEMM); scalesT (nullable, must be given
 *   together with qT): f32 [K/128][N/128], the same scales transposed.
 *   Requires N % 128 == 0 and K % 128 == 0.
 */
fp8bs_status fp8bs_quant_weight_128x128(const void *w_bf16, int64_t N,
                                        int64_t K, uint8_t *q, float *scales,
                                        uint8_t *qT, float *scalesT,
                                        fp8bs_stream_t stream);

/*
 * Backward-pass re-tiling [P1¶3]: cached FP8 activations quantized in 1x128
 * tiles become 128x1 tiles.  Each element is dequantized with one
 * round-to-nearest FP32 multiply, x_hat = decode(q) * s, and x_hat is
 * quantized again in groups of 128 consecutive rows of one column, written
 * transposed.
 *   q: E4M3 [M][K], scales: f32 [K/128][M]
 *   -> qT: E4M3 [K][M], scalesT: f32 [M/128][K].
 *   Requires M % 128 == 0 and K % 128 == 0.
 */
fp8bs_status fp8bs_requant_1x128_to_128x1(const uint8_t *q,
                                          const float *scales, int64_t M,
                                          int64_t K, uint8_t *qT,
                                          float *scalesT,
                                          fp8bs_stream_t stream);

/*
 * Block-scaled FP8 GEMM [P1¶2][P1¶3][P4¶4]: C = A * B^T with
 *   C[m][n] = sum over K-groups g of sa[g][m] * sB(n, g) * P_g[m][n],
 *   P_g[m][n] = sum_{k in g} A[m][k] * B[n][k]   (tensor cores, FP8 inputs),
 * each P_g promoted into an FP32 accumulator on the CUDA cores (one group =
 * 128 consecutive k).
 *   a: E4M3 [M][K], sa: f32 [K/128][M]
 *   b: E4M3 [N][K], sb: f32 [ceil(N/128)][K/128] (BLOCK) or [K/128][N]
 *   (TILE)
 *   c: [M][N], bf16 (round-to-nearest-even from FP32) or f32.
 *   Requires K % 128 == 0, N % 16 == 0, K > 0; M >= 0 (a ragged M tail is
 *   handled); M == 0 or N == 0 is a no-op.
 * Returns FP8BS_ERR_TIMEOUT only through fp8bs_get_device_error().
 * Every GEMM call is a programmatic dependent launch.  Its set-up (barriers,
 * tensor memory, tensor-map prefetch) may overlap the tail of the previous
 * kernel on `stream`, but it reads its inputs only after that kernel has
 * completed.  Stream order is unchanged for the caller.
 */
fp8bs_status fp8bs_gemm(const uint8_t *a, const float *sa, const uint8_t *b,
                        const float *sb, fp8bs_bscale_kind bkind, int64_t M,
                        int64_t N, int64_t K, void *c, fp8bs_out_dtype out,
                        fp8bs_stream_t stream);

/*
 * fp8bs_gemm with a choice of accumulation.  promote = 1 is fp8bs_gemm.
 * promote = 0 is the deliberately un-promoted variant used to measure what
 * tensor-core-only accumulation costs [P1¶4][P2¶3]: the whole K is
 * accumulated inside the tensor core and the scales are applied once at
 * the end, using K-group 0's scales (sa[0][m] and sB(n, 0)).  It is exact
 * only for operands whose scales are constant along K (row-wise
 * quantization); it is a measurement tool, not a second product path.
 */
fp8bs_status fp8bs_gemm_ex(const uint8_t *a, const float *sa,
                           const uint8_t *b, const float *sb,
                           fp8bs_bscale_kind bkind, int64_t M, int64_t N,
                           int64_t K, void *c, fp8bs_out_dtype out,
                           int promote, fp8bs_stream_t stream);

/*
 * Output tile shapes of the GEMM.  Every shape computes the same result;
 * they differ in speed.  FP8BS_TILE_AUTO (what fp8bs_gemm uses) picks, per
 * problem, the shape that needs the fewest full waves of tiles over the
 * device's SMs, weighted by each shape's efficiency.
 *   128xBN             one CTA per tile;
 *   256xBN_PAIR        a CTA pair (a cluster of two CTAs) whose tensor cores
 *                      compute one 256xBN tile together, each CTA loading
 *                      its own half of A and half of B (no copy is
 *                      multicast);
 *   ..._W12, ..._W16   the same with 12 or 16 promotion warps (8
 *                      otherwise), which read the tensor-core partial sums
 *                      out of tensor memory faster.
 */
typedef enum {
  FP8BS_TILE_AUTO = -1,
  FP8BS_TILE_128x128 = 0,
  FP8BS_TILE_128x256 = 1,
  FP8BS_TILE_256x128_PAIR = 2,
  FP8BS_TILE_256x160_PAIR = 3,
  FP8BS_TILE_256x192_PAIR = 4,
  FP8BS_TILE_256x224_PAIR = 5,
  FP8BS_TILE_256x256_PAIR = 6,
  FP8BS_TILE_256x192_PAIR_W12 = 7,
  FP8BS_TILE_256x256_PAIR_W16 = 8,
  FP8BS_TILE_256x192_PAIR_W16 = 9,
  FP8BS_TILE_256x128_PAIR_W16 = 10
} fp8bs_tile_shape;

/*
 * fp8bs_gemm_ex with an explicit tile shape (tuning and testing; every
 * shape must give results within the same tolerance).  An out-of-range
 * `tile` returns FP8BS_ERR_INVALID_ARG.
 */
fp8bs_status fp8bs_gemm_tiled(const uint8_t *a, const float *sa,
                              const uint8_t *b, const float *sb,
                              fp8bs_bscale_kind bkind, int64_t M, int64_t N,
                              int64_t K, void *c, fp8bs_out_dtype out,
                              int promote, fp8bs_tile_shape tile,
                              fp8bs_stream_t stream);

/*
 * fp8bs_gemm (promoted, every 128 K [P1¶3]) with stream-K scheduling of an
 * uneven last wave: when the last wave of whole output tiles would leave
 * the SMs idle for more than about half a wave (few tiles and long K, or
 * e.g. 3.03 or 6.05 waves), the K-groups of the last two waves' tiles (all
 * tiles, below two waves) are spread evenly over every SM.  The tile shape
 * is chosen with that plan in view, so it may differ from fp8bs_gemm's.  A tile split over several SMs is completed by the last
 * of them to finish: each writes its FP32 share of the tile to the
 * workspace, and the last sums the shares in K order (so the result does
 * not depend on which finishes last; it may differ from fp8bs_gemm's by
 * FP32 rounding, within the same tolerance) and writes C.
 * Other problems run exactly as fp8bs_gemm.
 *
 * fp8bs_gemm_streamk_workspace writes to *bytes the workspace size this
 * problem needs on the current device (0: no workspace, stream-K not used).
 * It launches nothing.  out: FP32 or BF16 only.
 *
 * fp8bs_gemm_streamk: arguments and layouts as fp8bs_gemm; workspace is
 * caller-owned device memory of at least that many bytes, 256-byte aligned
 * (FP8BS_ERR_MISALIGNED otherwise), not read or written by anything else
 * until the call's stream work is done.  Its contents need no
 * initialisation: the call zeroes the arrival counters on `stream` before
 * the GEMM.  A null workspace is accepted only when the problem needs none.
 * A workspace smaller than needed returns FP8BS_ERR_INVALID_ARG before any
 * launch.  Two calls in flight on one workspace race.
 */
fp8bs_status fp8bs_gemm_streamk_workspace(fp8bs_bscale_kind bkind, int64_t M,
                                          int64_t N, int64_t K,
                                          fp8bs_out_dtype out, size_t *bytes);
fp8bs_status fp8bs_gemm_streamk(const uint8_t *a, const float *sa,
                                const uint8_t *b, const float *sb,
                                fp8bs_bscale_kind bkind, int64_t M, int64_t N,
                                int64_t K, void *c, fp8bs_out_dtype out,
                                void *workspace, size_t workspace_bytes,
                                fp8bs_stream_t stream);

/*
 * fp8bs_gemm_streamk for callers that cannot allocate device memory: a
 * plain C host program with no device allocator of its own, or a runtime
 * that must not allocate once it is running (cudaMalloc can synchronize the
 * device and can fail under memory pressure).  The pages have no
 * counterpart to this call: it is a convenience of this library's API.
 * Arguments, layouts, result and error codes as fp8bs_gemm_streamk, without
 * the workspace: the stream-K shares and arrival counters live in one fixed
 * array of FP8BS_NOALLOC_SCRATCH_BYTES in the library's device memory, one
 * per device.  Nothing is allocated by the call.
 *   - A problem whose stream-K plan needs more scratch than that returns
 *     FP8BS_ERR_UNSUPPORTED_SHAPE before any launch
 *     (fp8bs_gemm_streamk_workspace gives the need).  Problems that plan no
 *     stream-K need none and run as fp8bs_gemm.
 *   - Nothing has to be zeroed by the caller: the array is zero when the
 *     library's module loads, the call zeroes the arrival counters on
 *     `stream` before each launch, and every share is written before it is
 *     read.
 *   - Set-up: the first call on each device that needs scratch looks up the
 *     array's address on that device (cudaGetSymbolAddress, with the device
 *     current) and may load the module; make that first call before
 *     beginning any stream capture.
 *   - One array per device: two calls in flight on one device (other
 *     streams, other host threads) race on it.  Order them on one stream or
 *     synchronize between them.
 */
#define FP8BS_NOALLOC_SCRATCH_BYTES (48u << 20)
fp8bs_status fp8bs_gemm_streamk_noalloc(const uint8_t *a, const float *sa,
                                        const uint8_t *b, const float *sb,
                                        fp8bs_bscale_kind bkind, int64_t M,
                                        int64_t N, int64_t K, void *c,
                                        fp8bs_out_dtype out,
                                        fp8bs_stream_t stream);

/*
 * Both operands of the forward GEMM quantized in one launch [P1¶3]: the
 * activation x in 1x128 tiles (exactly fp8bs_quant_act_1x128 with
 * transpose_out = 0) and the weight w in 128x128 blocks (exactly
 * fp8bs_quant_weight_128x128 without the transposed copy).  One launch pays
 * the launch, pipeline ramp and tail once for both tensors.
 *   x: bf16 [M][K] -> q: E4M3 [M][K], scales: f32 [K/128][M];
 *   w: bf16 [N][Kw] -> qw: E4M3 [N][Kw], w_scales: f32 [N/128][Kw/128].
 *   Requires K, N, Kw % 128 == 0 (M any); pointers 16-byte aligned.  An
 *   empty operand leaves the call to the other one.
 */
fp8bs_status fp8bs_quant_act_and_weight(const void *x_bf16, int64_t M,
                                        int64_t K, uint8_t *q, float *scales,
                                        const void *w_bf16, int64_t N,
                                        int64_t Kw, uint8_t *qw,
                                        float *w_scales, fp8bs_stream_t stream);

/*
 * E5M6 cache of an activation that the backward pass re-tiles from 1x128 to
 * 128x1 tiles [P1¶3: a custom E5M6 format is used only for these
 * activations].  Readings where the page is silent: E5M6 = sign, 5 exponent
 * bits (bias 15), 6 mantissa bits, exponent 0 = subnormals m * 2^-20,
 * exponent 31 = Inf/NaN, largest finite 65024 (code 0x7BF); rounding to
 * nearest even, saturating; NaN -> 0x7FF.  The cache keeps 1x128 tiles:
 * s = fl32(amax / 65024), code = E5M6(fl32(x / s)) (the rule of
 * fp8bs_quant_act_1x128 with 65024 in place of 448).  Codes are packed as a
 * little-endian 12-bit stream: element k of row m is bits 12k .. 12k+11 of
 * the row's 3K/2 bytes.
 *   x: bf16 [M][K] -> packed: [M][3K/2] bytes, scales: f32 [K/128][M].
 *   q, q_scales (both null or both set): also the E4M3 1x128 codes and
 *   scales of fp8bs_quant_act_1x128 for the forward GEMM, from the same read.
 *   Requires K % 128 == 0; pointers 16-byte aligned.  M == 0 or K == 0 is
 *   a no-op.
 */
fp8bs_status fp8bs_quant_act_e5m6(const void *x_bf16, int64_t M, int64_t K,
                                  uint8_t *packed, float *scales, uint8_t *q,
                                  float *q_scales, fp8bs_stream_t stream);

/*
 * The E5M6 cache re-tiled for the weight-gradient GEMM [P1¶3]: each element
 * is dequantized with one round-to-nearest multiply, x^ = fl32(decode(code)
 * * s), and the 128x1 rule of fp8bs_quant_act_1x128(transpose_out = 1) is
 * applied to x^.
 *   packed: [M][3K/2], scales: f32 [K/128][M] (fp8bs_quant_act_e5m6's
 *   output) -> qT: E4M3 [K][M], scalesT: f32 [M/128][K].
 *   Requires M % 128 == 0 and K % 128 == 0; pointers 16-byte aligned.
 */
fp8bs_status fp8bs_requant_e5m6_to_128x1(const uint8_t *packed,
                                         const float *scales, int64_t M,
                                         int64_t K, uint8_t *qT, float *scalesT,
                                         fp8bs_stream_t stream);

/*
 * Per-tensor FP8 quantization: the standard practice that the fine-grained
 * tiles replace [P1¶4][P3¶4] (one scale for the whole tensor, its max-abs
 * mapped to the FP8 maximum; sensitive to outliers).  Kept as the accuracy
 * baseline; the rule per element is that of fp8bs_quant_act_1x128 with a
 * single group: s = fl32(amax / 448), code = E4M3_RNE_satfinite(fl32(x / s)),
 * amax ignoring NaN.
 *   x: bf16 [rows][cols] -> q: E4M3 [rows][cols];
 *   scale: one float (device), written with s (it holds the running max
 *     while the call is in flight);
 *   scales_bcast (nullable when n_bcast == 0): n_bcast floats, each set to
 *     s, so q can go to fp8bs_gemm with any of its scale layouts (as A:
 *     [cols/128][rows]; as B with BLOCK scales: [rows/128][cols/128]).
 *   Requires cols % 16 == 0; x and q 16-byte aligned, scale and
 *   scales_bcast 4-byte aligned.  rows == 0 or cols == 0 is a no-op.
 *   Three launches and one 4-byte memset on `stream`; no scratch memory.
 */
fp8bs_status fp8bs_quant_per_tensor(const void *x_bf16, int64_t rows,
                                    int64_t cols, uint8_t *q, float *scale,
                                    float *scales_bcast, int64_t n_bcast,
                                    fp8bs_stream_t stream);

/*
 * The block-scaled GEMM with its output quantized in the epilogue, for the
 * next layer [P2¶1: the BF16 result otherwise makes a round trip through HBM
 * before it is quantized].  Computes the FP32 C of fp8bs_gemm (promoted),
 * then quantizes each 1x128 tile of each C row by the rule of
 * fp8bs_quant_act_1x128 applied to the FP32 values: s = fl32(amax / 448),
 * code = E4M3_RNE_satfinite(fl32(C / s)).
 *   c: E4M3 [M][N], c_scales: f32 [N/128][M] (the layout of
 *   fp8bs_quant_act_1x128's output, so c can feed the next GEMM as its A).
 *   Requires N % 128 == 0 (and the fp8bs_gemm requirements); always uses
 *   256 x 256 CTA-pair tiles.
 */
fp8bs_status fp8bs_gemm_quant_out(const uint8_t *a, const float *sa,
                                  const uint8_t *b, const float *sb,
                                  fp8bs_bscale_kind bkind, int64_t M,
                                  int64_t N, int64_t K, uint8_t *c,
                                  float *c_scales, fp8bs_stream_t stream);

/* Static English name of a status code. */
const char *fp8bs_status_string(fp8bs_status status);

/*
 * Reports and clears the device error words that bounded waits inside the
 * kernels set when they give up (FP8BS_ERR_TIMEOUT), or FP8BS_ERR_CUDA if a
 * CUDA call failed.  The words are per device and shared by every stream and
 * host thread: a kernel that timed out on any stream sets them.  The query
 * takes them in stream order on `stream` with an atomic exchange (one
 * one-thread kernel per word), then synchronizes `stream`, so each timeout
 * is reported by exactly one query and none is lost.  To attribute a
 * timeout to one stream, query after a device-wide synchronization.  The
 * first query from a host thread allocates two mapped pinned host words for
 * that thread, kept until the process exits.
 */
fp8bs_status fp8bs_get_device_error(fp8bs_stream_t stream);

/* cudaError_t value of the last CUDA failure seen by this host thread
 * (FP8BS_ERR_CUDA leaves the detail here; 0 if none). */
int fp8bs_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int fp8bs_version(void);

/*
 * TEST SUPPORT ONLY -- exercises the GEMM's bounded waits without faulting
 * or hanging the GPU.  Runs fp8bs_gemm_tiled (BLOCK scales, FP32 out,
 * promoted, the given tile shape) except that the TMA producer skips
 * pipeline iteration `skip_iter` (>= 0): its copy is never issued and its
 * mbarrier never completes, so the consumer waiting on it gives up after its
 * time limit (about 2 s), every warp winds down, TMEM is freed and the
 * kernel returns.  The C output is then undefined; fp8bs_get_device_error()
 * reports FP8BS_ERR_TIMEOUT and clears the error word, after which the
 * context is usable as before.
 */
fp8bs_status fp8bs_debug_gemm_stall(const uint8_t *a, const float *sa,
                                    const uint8_t *b, const float *sb,
                                    int64_t M, int64_t N, int64_t K, void *c,
                                    int skip_iter, fp8bs_tile_shape tile,
                                    fp8bs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
