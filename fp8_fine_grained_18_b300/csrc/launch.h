// launch.h -- internal host-side launchers of the libfp8bs kernels.  The
// exported C ABI (include/fp8bs.h) validates arguments and calls these.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8bs {

// Tensor map of a dense row-major matrix [rows][cols] of 1-, 2- or 4-byte
// elements, box of box_cols x box_rows elements, optionally with the 128-byte
// swizzle; out-of-range elements read as zero.  False if encoding failed.
bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, int64_t rows, int64_t cols,
                  int box_cols, int box_rows, bool swizzle128);

cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                   cudaStream_t stream);
cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, uint8_t* qT, float* sT,
                                   cudaStream_t stream);
cudaError_t launch_quant_act_dual(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                  uint8_t* qT, float* sT, cudaStream_t stream);
// Q1 of x [M][K] and Q2 of w [N][Kw] in one launch (same outputs as the two
// launchers above).
cudaError_t launch_quant_act_and_weight(const void* x, int64_t M, int64_t K, uint8_t* q,
                                        float* s, const void* w, int64_t N, int64_t Kw,
                                        uint8_t* qw, float* sw, cudaStream_t stream);
cudaError_t launch_quant_weight_128x128(const void* w, int64_t N, int64_t K, uint8_t* q, float* s,
                                        uint8_t* qT, float* sT, cudaStream_t stream);
// Per-tensor scale of n bf16 values (n % 8 == 0): q codes, *scale, and
// n_bcast copies of the scale in bcast (nullable when n_bcast == 0).
cudaError_t launch_quant_per_tensor(const void* x, int64_t n, uint8_t* q, float* scale,
                                    float* bcast, int64_t n_bcast, cudaStream_t stream);
// E5M6 cache (packed [M][3K/2], scales [K/128][M]) of a bf16 activation,
// with its E4M3 1x128 codes from the same read when q is non-null.
cudaError_t launch_quant_act_e5m6(const void* x, int64_t M, int64_t K, uint8_t* e5, float* s5,
                                  uint8_t* q, float* s, cudaStream_t stream);
// The E5M6 cache re-tiled to 128x1 E4M3 tiles, transposed (M % 128 == 0).
cudaError_t launch_requant_e5m6_to_128x1(const uint8_t* e5, const float* s5, int64_t M, int64_t K,
                                         uint8_t* qT, float* sT, cudaStream_t stream);
cudaError_t launch_requant_1x128_to_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                          uint8_t* qT, float* sT, cudaStream_t stream);

struct GemmArgs {
  const uint8_t* a;
  const float* sa;
  const uint8_t* b;
  const float* sb;
  bool b_tile;  // B scales per 1x128 tile (else per 128x128 block)
  int64_t M, N, K;
  void* c;
  float* c_scales;  // E4M3 output only: [N/128][M]
  int out;          // 0 FP32, 1 BF16, 2 E4M3 codes + 1x128 scales
  bool promote;
  int skip_iter;  // test hook: producer skips this pipeline iteration (-1: never)
  int tile;       // fp8bs_tile_shape value; -1 chooses per problem shape
  // Stream-K workspace (device memory, 256-byte aligned) and its size; null
  // runs every unit whole.  With ws_need set, nothing is launched: the
  // workspace bytes this problem needs are written there (0: stream-K is not
  // used for it).
  void* ws = nullptr;
  size_t ws_bytes = 0;
  size_t* ws_need = nullptr;
};

cudaError_t launch_gemm(const GemmArgs& args, cudaStream_t stream);

// The fixed scratch of fp8bs_gemm_streamk_noalloc on the current device (its
// address is looked up once per device) and its size.
cudaError_t noalloc_scratch(void** ptr, size_t* bytes);
size_t noalloc_scratch_bytes();

// Enqueue on `stream` a one-thread kernel that atomically exchanges the
// device error word of the bounded waits in the GEMM (or in the quantizers)
// with 0 and writes the old value to *dst (device-visible memory, e.g. a
// mapped pinned host word).  0 means nothing timed out.
cudaError_t enqueue_take_gemm_error(unsigned int* dst, cudaStream_t stream);
cudaError_t enqueue_take_quant_error(unsigned int* dst, cudaStream_t stream);

}  // namespace fp8bs
