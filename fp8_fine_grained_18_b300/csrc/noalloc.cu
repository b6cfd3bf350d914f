// noalloc.cu -- scratch for fp8bs_gemm_streamk_noalloc: the stream-K GEMM
// for callers that cannot allocate device memory.  Its workspace is one
// fixed array of this module's device memory instead of a caller buffer.
#include <mutex>

#include <cuda_runtime.h>

#include "launch.h"

namespace fp8bs {
namespace {

// 48 MiB: room for every stream-K workspace on 148 SMs (at most about
// 38.8 MB: two FP32 shares of a 128 x 256 accumulator per CTA, and the
// arrival counters); plans that need more (devices with more SMs) are
// refused by the entry point.  The array is zero when the module loads.
// The CUDA runtime places it when this module is loaded: on first use under
// lazy module loading (the default), at context creation otherwise.
constexpr size_t kScratchBytes = size_t(48) << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct DeviceScratch {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceScratch g_dev[kMaxDevices];

}  // namespace

cudaError_t noalloc_scratch(void** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceScratch& d = g_dev[dev];
  // once per device, with that device current: the array's address in it
  std::call_once(d.once, [&d] { d.err = cudaGetSymbolAddress(&d.ptr, g_scratch); });
  if (d.err != cudaSuccess) return d.err;
  *ptr = d.ptr;
  *bytes = kScratchBytes;
  return cudaSuccess;
}

size_t noalloc_scratch_bytes() { return kScratchBytes; }

}  // namespace fp8bs
