// api.cu -- the exported C ABI of libfp8bs (declared in include/fp8bs.h):
// host-side argument validation, device-architecture check, and dispatch to
// the kernel launchers.  Nothing is launched when an argument is invalid.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/fp8bs.h"
#include "launch.h"

namespace {

thread_local int t_last_cuda_error = 0;
thread_local unsigned int* t_err_words = nullptr;  // see fp8bs_get_device_error

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

fp8bs_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FP8BS_OK;
  t_last_cuda_error = (int)e;
  return FP8BS_ERR_CUDA;
}

// 0 = unknown, 1 = sm_103, 2 = other (several host threads may fill it)
std::atomic<int> g_arch_cache[128];

fp8bs_status check_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_status(e);
  }
  int cached = (dev >= 0 && dev < 128) ? g_arch_cache[dev].load() : 0;
  if (cached == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      return cuda_status(cudaGetLastError());
    }
    cached = (major == 10 && minor == 3) ? 1 : 2;
    if (dev >= 0 && dev < 128) g_arch_cache[dev].store(cached);
  }
  return cached == 1 ? FP8BS_OK : FP8BS_ERR_ARCH;
}

cudaStream_t as_cuda(fp8bs_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

constexpr int64_t kMaxDim = (int64_t)1 << 31;  // kernels index rows with int32

// The transposing quantizers index 128 x 128 tiles, rows, columns and the
// packed E5M6 row bytes (1.5 K) with int32.
bool transposed_shape_ok(int64_t M, int64_t K) {
  return M < ((int64_t)1 << 30) && K < ((int64_t)1 << 30) &&
         (M / 128) * (K / 128) < ((int64_t)1 << 31);
}

fp8bs_status gemm_common(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                         fp8bs_bscale_kind bkind, int64_t M, int64_t N, int64_t K, void* c,
                         fp8bs_out_dtype out, int promote, int skip_iter, int tile,
                         fp8bs_stream_t stream, float* c_scales = nullptr, void* ws = nullptr,
                         size_t ws_bytes = 0) {
  if (M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (bkind != FP8BS_BSCALE_BLOCK_128x128 && bkind != FP8BS_BSCALE_TILE_1x128)
    return FP8BS_ERR_INVALID_ARG;
  if (out != FP8BS_OUT_BF16 && out != FP8BS_OUT_F32 && out != FP8BS_OUT_E4M3_1x128)
    return FP8BS_ERR_INVALID_ARG;
  if (out == FP8BS_OUT_E4M3_1x128 && (promote != 1 || !c_scales)) return FP8BS_ERR_INVALID_ARG;
  if (promote != 0 && promote != 1) return FP8BS_ERR_INVALID_ARG;
  if (tile < FP8BS_TILE_AUTO || tile > FP8BS_TILE_256x128_PAIR_W16) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FP8BS_OK;
  if (!a || !sa || !b || !sb || !c) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N % 16 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (out == FP8BS_OUT_E4M3_1x128 && N % 128 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(c) ||
      (c_scales && !aligned16(c_scales)))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  fp8bs::GemmArgs g;
  g.a = a;
  g.sa = sa;
  g.b = b;
  g.sb = sb;
  g.b_tile = bkind == FP8BS_BSCALE_TILE_1x128;
  g.M = M;
  g.N = N;
  g.K = K;
  g.c = c;
  g.c_scales = c_scales;
  g.out = out == FP8BS_OUT_BF16 ? 1 : out == FP8BS_OUT_E4M3_1x128 ? 2 : 0;
  g.promote = promote != 0;
  g.skip_iter = skip_iter;
  g.tile = tile;
  if (ws != nullptr) {
    size_t need = 0;
    g.ws_need = &need;
    fp8bs_status qs = cuda_status(fp8bs::launch_gemm(g, as_cuda(stream)));
    if (qs != FP8BS_OK) return qs;
    if (ws_bytes < need) return FP8BS_ERR_INVALID_ARG;
    if (need > 0 && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FP8BS_ERR_MISALIGNED;
    g.ws_need = nullptr;
    g.ws = ws;
    g.ws_bytes = ws_bytes;
  }
  return cuda_status(fp8bs::launch_gemm(g, as_cuda(stream)));
}

// Workspace bytes of the stream-K GEMM for this problem on the current
// device (shape checks as gemm_common; no pointers needed).
fp8bs_status streamk_need(fp8bs_bscale_kind bkind, int64_t M, int64_t N, int64_t K,
                          fp8bs_out_dtype out, size_t* bytes) {
  if (!bytes) return FP8BS_ERR_INVALID_ARG;
  *bytes = 0;
  if (M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (bkind != FP8BS_BSCALE_BLOCK_128x128 && bkind != FP8BS_BSCALE_TILE_1x128)
    return FP8BS_ERR_INVALID_ARG;
  if (out != FP8BS_OUT_BF16 && out != FP8BS_OUT_F32) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FP8BS_OK;
  if (K == 0 || K % 128 != 0 || N % 16 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  fp8bs::GemmArgs g;
  g.a = nullptr;
  g.sa = nullptr;
  g.b = nullptr;
  g.sb = nullptr;
  g.b_tile = bkind == FP8BS_BSCALE_TILE_1x128;
  g.M = M;
  g.N = N;
  g.K = K;
  g.c = nullptr;
  g.c_scales = nullptr;
  g.out = out == FP8BS_OUT_BF16 ? 1 : 0;
  g.promote = true;
  g.skip_iter = -1;
  g.tile = FP8BS_TILE_AUTO;
  g.ws_need = bytes;
  return cuda_status(fp8bs::launch_gemm(g, nullptr));
}

}  // namespace

extern "C" {

fp8bs_status fp8bs_quant_act_1x128(const void* x_bf16, int64_t M, int64_t K, int transpose_out,
                                   uint8_t* q, float* scales, fp8bs_stream_t stream) {
  if (M < 0 || K < 0 || (transpose_out != 0 && transpose_out != 1)) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return FP8BS_OK;
  if (!x_bf16 || !q || !scales) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0 || (transpose_out && M % 128 != 0)) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (K / 128 > 65535 || M >= kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (transpose_out && !transposed_shape_ok(M, K)) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_bf16) || !aligned16(q) || !aligned16(scales)) return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  cudaError_t e = transpose_out
                      ? fp8bs::launch_quant_act_128x1(x_bf16, M, K, q, scales, as_cuda(stream))
                      : fp8bs::launch_quant_act_1x128(x_bf16, M, K, q, scales, as_cuda(stream));
  return cuda_status(e);
}

fp8bs_status fp8bs_quant_act_dual(const void* x_bf16, int64_t M, int64_t K, uint8_t* q,
                                  float* scales, uint8_t* qT, float* scalesT,
                                  fp8bs_stream_t stream) {
  if (M < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return FP8BS_OK;
  if (!x_bf16 || !q || !scales || !qT || !scalesT) return FP8BS_ERR_INVALID_ARG;
  if (M % 128 != 0 || K % 128 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!transposed_shape_ok(M, K)) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_bf16) || !aligned16(q) || !aligned16(scales) || !aligned16(qT) ||
      !aligned16(scalesT))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  return cuda_status(
      fp8bs::launch_quant_act_dual(x_bf16, M, K, q, scales, qT, scalesT, as_cuda(stream)));
}

fp8bs_status fp8bs_quant_weight_128x128(const void* w_bf16, int64_t N, int64_t K, uint8_t* q,
                                        float* scales, uint8_t* qT, float* scalesT,
                                        fp8bs_stream_t stream) {
  if (N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if ((qT == nullptr) != (scalesT == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return FP8BS_OK;
  if (!w_bf16 || !q || !scales) return FP8BS_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (N / 128 > 65535 || K / 128 > (int64_t)1 << 30) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w_bf16) || !aligned16(q) || !aligned16(scales) || (qT && !aligned16(qT)) ||
      (scalesT && !aligned16(scalesT)))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  return cuda_status(
      fp8bs::launch_quant_weight_128x128(w_bf16, N, K, q, scales, qT, scalesT, as_cuda(stream)));
}

fp8bs_status fp8bs_quant_per_tensor(const void* x_bf16, int64_t rows, int64_t cols, uint8_t* q,
                                    float* scale, float* scales_bcast, int64_t n_bcast,
                                    fp8bs_stream_t stream) {
  if (rows < 0 || cols < 0 || n_bcast < 0) return FP8BS_ERR_INVALID_ARG;
  if (n_bcast > 0 && !scales_bcast) return FP8BS_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP8BS_OK;
  if (!x_bf16 || !q || !scale) return FP8BS_ERR_INVALID_ARG;
  if (cols % 16 != 0 || rows >= kMaxDim * 64 || cols >= kMaxDim * 64 ||
      rows > ((int64_t)1 << 40) / cols || n_bcast > ((int64_t)1 << 40))
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_bf16) || !aligned16(q) || !aligned4(scale) ||
      (scales_bcast && !aligned4(scales_bcast)))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  return cuda_status(fp8bs::launch_quant_per_tensor(x_bf16, rows * cols, q, scale, scales_bcast,
                                                    n_bcast, as_cuda(stream)));
}

fp8bs_status fp8bs_quant_act_e5m6(const void* x_bf16, int64_t M, int64_t K, uint8_t* packed,
                                  float* scales, uint8_t* q, float* q_scales,
                                  fp8bs_stream_t stream) {
  if (M < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if ((q == nullptr) != (q_scales == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return FP8BS_OK;
  if (!x_bf16 || !packed || !scales) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (K / 128 > 65535 || M >= kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_bf16) || !aligned16(packed) || !aligned16(scales) || (q && !aligned16(q)) ||
      (q_scales && !aligned16(q_scales)))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  return cuda_status(
      fp8bs::launch_quant_act_e5m6(x_bf16, M, K, packed, scales, q, q_scales, as_cuda(stream)));
}

fp8bs_status fp8bs_requant_e5m6_to_128x1(const uint8_t* packed, const float* scales, int64_t M,
                                         int64_t K, uint8_t* qT, float* scalesT,
                                         fp8bs_stream_t stream) {
  if (M < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return FP8BS_OK;
  if (!packed || !scales || !qT || !scalesT) return FP8BS_ERR_INVALID_ARG;
  if (M % 128 != 0 || K % 128 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!transposed_shape_ok(M, K)) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(packed) || !aligned16(scales) || !aligned16(qT) || !aligned16(scalesT))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  return cuda_status(
      fp8bs::launch_requant_e5m6_to_128x1(packed, scales, M, K, qT, scalesT, as_cuda(stream)));
}

fp8bs_status fp8bs_quant_act_and_weight(const void* x_bf16, int64_t M, int64_t K, uint8_t* q,
                                        float* scales, const void* w_bf16, int64_t N, int64_t Kw,
                                        uint8_t* qw, float* w_scales, fp8bs_stream_t stream) {
  if (M < 0 || K < 0 || N < 0 || Kw < 0) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || K == 0)
    return fp8bs_quant_weight_128x128(w_bf16, N, Kw, qw, w_scales, nullptr, nullptr, stream);
  if (N == 0 || Kw == 0) return fp8bs_quant_act_1x128(x_bf16, M, K, 0, q, scales, stream);
  if (!x_bf16 || !q || !scales || !w_bf16 || !qw || !w_scales) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 128 != 0 || Kw % 128 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  const int64_t tiles = ((M + 127) / 128) * (K / 128) + (N / 128) * (Kw / 128);
  if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim || Kw >= kMaxDim || tiles >= kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_bf16) || !aligned16(q) || !aligned16(scales) || !aligned16(w_bf16) ||
      !aligned16(qw) || !aligned16(w_scales))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  return cuda_status(fp8bs::launch_quant_act_and_weight(x_bf16, M, K, q, scales, w_bf16, N, Kw,
                                                        qw, w_scales, as_cuda(stream)));
}

fp8bs_status fp8bs_requant_1x128_to_128x1(const uint8_t* q, const float* scales, int64_t M,
                                          int64_t K, uint8_t* qT, float* scalesT,
                                          fp8bs_stream_t stream) {
  if (M < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return FP8BS_OK;
  if (!q || !scales || !qT || !scalesT) return FP8BS_ERR_INVALID_ARG;
  if (M % 128 != 0 || K % 128 != 0) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!transposed_shape_ok(M, K)) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(q) || !aligned16(scales) || !aligned16(qT) || !aligned16(scalesT))
    return FP8BS_ERR_MISALIGNED;
  fp8bs_status st = check_device();
  if (st != FP8BS_OK) return st;
  return cuda_status(
      fp8bs::launch_requant_1x128_to_128x1(q, scales, M, K, qT, scalesT, as_cuda(stream)));
}

fp8bs_status fp8bs_gemm(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                        fp8bs_bscale_kind bkind, int64_t M, int64_t N, int64_t K, void* c,
                        fp8bs_out_dtype out, fp8bs_stream_t stream) {
  return gemm_common(a, sa, b, sb, bkind, M, N, K, c, out, 1, -1, FP8BS_TILE_AUTO, stream);
}

fp8bs_status fp8bs_gemm_ex(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                           fp8bs_bscale_kind bkind, int64_t M, int64_t N, int64_t K, void* c,
                           fp8bs_out_dtype out, int promote, fp8bs_stream_t stream) {
  return gemm_common(a, sa, b, sb, bkind, M, N, K, c, out, promote, -1, FP8BS_TILE_AUTO,
                     stream);
}

fp8bs_status fp8bs_gemm_tiled(const uint8_t* a, const float* sa, const uint8_t* b,
                              const float* sb, fp8bs_bscale_kind bkind, int64_t M, int64_t N,
                              int64_t K, void* c, fp8bs_out_dtype out, int promote,
                              fp8bs_tile_shape tile, fp8bs_stream_t stream) {
  return gemm_common(a, sa, b, sb, bkind, M, N, K, c, out, promote, -1, tile, stream);
}

fp8bs_status fp8bs_gemm_streamk_workspace(fp8bs_bscale_kind bkind, int64_t M, int64_t N,
                                          int64_t K, fp8bs_out_dtype out, size_t* bytes) {
  return streamk_need(bkind, M, N, K, out, bytes);
}

fp8bs_status fp8bs_gemm_streamk(const uint8_t* a, const float* sa, const uint8_t* b,
                                const float* sb, fp8bs_bscale_kind bkind, int64_t M, int64_t N,
                                int64_t K, void* c, fp8bs_out_dtype out, void* workspace,
                                size_t workspace_bytes, fp8bs_stream_t stream) {
  if (out != FP8BS_OUT_BF16 && out != FP8BS_OUT_F32) return FP8BS_ERR_INVALID_ARG;
  if (workspace == nullptr && workspace_bytes != 0) return FP8BS_ERR_INVALID_ARG;
  if (workspace == nullptr) {
    // no workspace: valid only where the plan needs none
    size_t need = 0;
    fp8bs_status st = streamk_need(bkind, M, N, K, out, &need);
    if (st != FP8BS_OK) return st;
    if (need > 0) return FP8BS_ERR_INVALID_ARG;
  }
  return gemm_common(a, sa, b, sb, bkind, M, N, K, c, out, 1, -1, FP8BS_TILE_AUTO, stream,
                     nullptr, workspace, workspace_bytes);
}

fp8bs_status fp8bs_gemm_streamk_noalloc(const uint8_t* a, const float* sa, const uint8_t* b,
                                        const float* sb, fp8bs_bscale_kind bkind, int64_t M,
                                        int64_t N, int64_t K, void* c, fp8bs_out_dtype out,
                                        fp8bs_stream_t stream) {
  if (out != FP8BS_OUT_BF16 && out != FP8BS_OUT_F32) return FP8BS_ERR_INVALID_ARG;
  size_t need = 0;
  fp8bs_status st = streamk_need(bkind, M, N, K, out, &need);
  if (st != FP8BS_OK) return st;
  if (need > fp8bs::noalloc_scratch_bytes()) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    cudaError_t e = fp8bs::noalloc_scratch(&ws, &ws_bytes);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return gemm_common(a, sa, b, sb, bkind, M, N, K, c, out, 1, -1, FP8BS_TILE_AUTO, stream,
                     nullptr, ws, ws_bytes);
}

fp8bs_status fp8bs_gemm_quant_out(const uint8_t* a, const float* sa, const uint8_t* b,
                                   const float* sb, fp8bs_bscale_kind bkind, int64_t M, int64_t N,
                                   int64_t K, uint8_t* c, float* c_scales,
                                   fp8bs_stream_t stream) {
  return gemm_common(a, sa, b, sb, bkind, M, N, K, c, FP8BS_OUT_E4M3_1x128, 1, -1,
                     FP8BS_TILE_AUTO, stream, c_scales);
}

fp8bs_status fp8bs_debug_gemm_stall(const uint8_t* a, const float* sa, const uint8_t* b,
                                    const float* sb, int64_t M, int64_t N, int64_t K, void* c,
                                    int skip_iter, fp8bs_tile_shape tile, fp8bs_stream_t stream) {
  if (skip_iter < 0) return FP8BS_ERR_INVALID_ARG;
  return gemm_common(a, sa, b, sb, FP8BS_BSCALE_BLOCK_128x128, M, N, K, c, FP8BS_OUT_F32, 1,
                     skip_iter, tile, stream);
}

const char* fp8bs_status_string(fp8bs_status s) {
  switch (s) {
    case FP8BS_OK: return "ok";
    case FP8BS_ERR_INVALID_ARG: return "invalid argument";
    case FP8BS_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FP8BS_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FP8BS_ERR_ARCH: return "device is not sm_103 (B300)";
    case FP8BS_ERR_CUDA: return "CUDA error";
    case FP8BS_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

fp8bs_status fp8bs_get_device_error(fp8bs_stream_t stream) {
  // Two mapped pinned host words per calling host thread, allocated on its
  // first query and kept until the process exits.  The device writes the
  // taken error words there in stream order; the host reads them after the
  // stream synchronization.
  if (!t_err_words) {
    void* p = nullptr;
    cudaError_t e =
        cudaHostAlloc(&p, 2 * sizeof(unsigned int), cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_status(e);
    t_err_words = static_cast<unsigned int*>(p);
  }
  volatile unsigned int* w = t_err_words;
  w[0] = 0u;
  w[1] = 0u;
  unsigned int* dptr = nullptr;
  cudaError_t e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&dptr), t_err_words, 0);
  if (e != cudaSuccess) return cuda_status(e);
  e = fp8bs::enqueue_take_gemm_error(dptr, as_cuda(stream));
  if (e != cudaSuccess) return cuda_status(e);
  e = fp8bs::enqueue_take_quant_error(dptr + 1, as_cuda(stream));
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaStreamSynchronize(as_cuda(stream));
  if (e != cudaSuccess) return cuda_status(e);
  return (w[0] | w[1]) ? FP8BS_ERR_TIMEOUT : FP8BS_OK;
}

int fp8bs_last_cuda_error(void) { return t_last_cuda_error; }

int fp8bs_version(void) { return 100; }

}  // extern "C"
