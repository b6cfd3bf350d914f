// gemm.cu -- block-scaled FP8 GEMM for sm_103a with FP32 promotion.
//
// C[m][n] = sum_g sa[g][m] * sB(n, g) * P_g[m][n],   P_g = A_g * B_g^T,
// where g runs over 128-wide K groups (DeepSeek-V3 fine-grained FP8 GEMM:
// per-group scales along K multiplied in on the CUDA cores while
// dequantizing, page P1 paragraph 2; partial sums promoted to FP32 because
// tensor-core accumulation alone is limited, P1 paragraphs 3-4, P2
// paragraph 3; FP8 in, BF16/FP32 out, P4 paragraph 4).
//
// B300 design (the pages' H800 WGMMA kernel is prior art only):
//   * persistent CTAs, one per SM, 128 x BN output tiles;
//   * warp 0 -- TMA producer: A and B K-group tiles (128 B rows, 128-byte
//     swizzle) into an STAGES-deep shared-memory ring (mbarrier full/empty);
//   * warp 1 -- MMA issuer: per K-group, four tcgen05.mma kind::f8f6f4
//     (K = 32 each) into one of TBUF TMEM partial buffers, then
//     tcgen05.commit to free the smem stage and to publish the partial;
//   * warp 2 -- scale loader: the K-group's 128 row scales of A and the
//     tile's B scales into a small shared ring;
//   * warps 4..11 -- promotion: each owns 32 TMEM lanes (rows) and half the
//     tile's columns, keeps the FP32 accumulator in registers, and per
//     K-group does acc += P_g * (sa * sb) while the tensor core already
//     computes the next group's partial into the other TMEM buffer (the
//     "overlapping of the two operations" of P3 paragraph 4 / P4 paragraph 1);
//     the epilogue converts to BF16 (RNE) or keeps FP32 and stores.
//   * every mbarrier wait is bounded (globaltimer); on expiry the kernel
//     sets a device error word and an abort flag, every role winds down,
//     in-flight copies and MMAs are drained (bounded) and TMEM is freed.
//
// The un-promoted variant (PROMOTE = false) keeps the whole K inside one
// TMEM accumulator and applies K-group 0's scales once at the end: the
// measurement of what tensor-core-only accumulation costs (P1 paragraph 4).
#include <cuda.h>
#include <cuda_bf16.h>

#include "fp8_common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace fp8bs {

__device__ unsigned int g_device_error;

namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;            // one scale group per pipeline stage
constexpr int kThreads = 384;       // 12 warps
constexpr int kFirstPromoWarp = 4;  // warps 4..11
constexpr int kPromoWarps = 8;
constexpr int kScaleSlots = 8;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

enum : unsigned int {
  kErrProducer = 1u,
  kErrMma = 2u,
  kErrScales = 4u,
  kErrPromo = 8u,
  kErrDrain = 16u,
};

struct Params {
  const float* sa;
  const float* sb;
  void* c;
  int M, N, K, KB;
  int num_m_tiles, num_tiles;
  int skip_iter;
};

// Bounded wait.  Returns false when this wait expired (the error word and
// the CTA's abort flag get set) or another role already aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int site) {
  const uint32_t addr = ptx::smem_addr(bar);
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (ptx::mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(addr, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      atomicOr(&g_device_error, site);
      return false;
    }
  }
}

template <int BN, int STAGES, int TBUF>
struct Smem {
  static constexpr int kABytes = kBM * kBK;          // 16 KB
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kScaleB = BN + 4;             // B scales per slot
  static constexpr int kScaleFloats = kBM + kScaleB;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffScale = kOffB + STAGES * kBBytes;
  static constexpr int kOffBar = kOffScale + kScaleSlots * kScaleFloats * 4;
  static constexpr int kNumBars = 2 * STAGES + 2 * TBUF + 2 * kScaleSlots + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

__host__ __device__ constexpr int tmem_cols_for(int cols) {
  return cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
}

template <int BN, int STAGES, int TBUF, bool PROMOTE, bool OUT_BF16, bool B_TILE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, const Params p) {
  using L = Smem<BN, STAGES, TBUF>;
  static_assert(BN % 64 == 0 && BN <= 256, "BN");
  static_assert(BN * TBUF <= 512, "TMEM");
  constexpr int kHalf = BN / 2;        // columns per promotion warp
  constexpr int kChunks = kHalf / 32;  // 32-column TMEM loads per warp
  constexpr int kChunksPerRound = kChunks < 2 ? kChunks : 2;
  constexpr uint32_t kTmemCols = tmem_cols_for(BN * TBUF);
  constexpr uint32_t kIdesc = ptx::idesc_e4m3_f32(kBM, BN);
  constexpr uint32_t kStageTx = L::kABytes + L::kBBytes;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + L::kOffA;
  uint8_t* sB = smem + L::kOffB;
  float* sScale = reinterpret_cast<float*>(smem + L::kOffScale);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + TBUF;
  uint64_t* sfull = tempty + TBUF;
  uint64_t* sempty = sfull + kScaleSlots;
  uint64_t* drain = sempty + kScaleSlots;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < TBUF; ++i) {
      ptx::mbar_init(&tfull[i], 1);
      ptx::mbar_init(&tempty[i], kPromoWarps);
    }
    for (int i = 0; i < kScaleSlots; ++i) {
      ptx::mbar_init(&sfull[i], 32);
      ptx::mbar_init(&sempty[i], kPromoWarps);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_base_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_base_slot;

  const int KB = p.KB;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_a);
      ptx::prefetch_tmap(&tmap_b);
      uint32_t it = 0;
      uint32_t issued_mask = 0;  // stages with a copy issued at least once
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1;
          if (!wait_bar(&empty[stage], phase ^ 1, abort_flag, kErrProducer)) { ok = false; break; }
          if ((int)it == p.skip_iter) continue;  // test hook: never arrives
          ptx::mbar_arrive_expect_tx(&full[stage], kStageTx);
          ptx::tma_load_2d(sA + stage * L::kABytes, &tmap_a, &full[stage], kb * kBK, mt * kBM);
          ptx::tma_load_2d(sB + stage * L::kBBytes, &tmap_b, &full[stage], kb * kBK, nt * BN);
          issued_mask |= 1u << stage;
        }
      }
      // Drain: wait (bounded) until the last copy issued into each stage has
      // landed, so no copy is in flight when the CTA exits.
      const uint32_t last = it;
      for (uint32_t s = 0; s < STAGES; ++s) {
        if (!(issued_mask & (1u << s)) || last == 0) continue;
        // the last iteration index < last that used stage s
        uint32_t li = (last - 1) - (((last - 1) % STAGES + STAGES - s) % STAGES);
        if ((int)li == p.skip_iter) continue;
        const uint32_t addr = ptx::smem_addr(&full[s]);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(addr, (li / STAGES) & 1)) {
          if (ptx::globaltimer() - t0 > kTimeoutNs) { atomicOr(&g_device_error, kErrDrain); break; }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, kt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        if (PROMOTE) {
          for (int kb = 0; kb < KB; ++kb, ++it, ++kt) {
            const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
            if (!wait_bar(&tempty[buf], tph ^ 1, abort_flag, kErrMma)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1;
            if (!wait_bar(&full[stage], phase, abort_flag, kErrMma)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t a0 = ptx::smem_addr(sA + stage * L::kABytes);
            const uint32_t b0 = ptx::smem_addr(sB + stage * L::kBBytes);
            const uint32_t d = tmem_base + buf * BN;
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k)
              ptx::mma_f8f6f4(d, ptx::smem_desc_k128_sw128(a0 + 32 * k),
                              ptx::smem_desc_k128_sw128(b0 + 32 * k), kIdesc, k > 0);
            ptx::tc_commit(&empty[stage]);
            ptx::tc_commit(&tfull[buf]);
          }
        } else {
          const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
          if (!wait_bar(&tempty[buf], tph ^ 1, abort_flag, kErrMma)) break;
          ptx::tc_fence_after();
          const uint32_t d = tmem_base + buf * BN;
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1;
            if (!wait_bar(&full[stage], phase, abort_flag, kErrMma)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t a0 = ptx::smem_addr(sA + stage * L::kABytes);
            const uint32_t b0 = ptx::smem_addr(sB + stage * L::kBBytes);
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k)
              ptx::mma_f8f6f4(d, ptx::smem_desc_k128_sw128(a0 + 32 * k),
                              ptx::smem_desc_k128_sw128(b0 + 32 * k), kIdesc,
                              (kb > 0 || k > 0) ? 1u : 0u);
            ptx::tc_commit(&empty[stage]);
          }
          if (!ok) break;
          ptx::tc_commit(&tfull[buf]);
          ++kt;
        }
      }
      // Drain: every MMA this thread issued has completed before TMEM is freed.
      ptx::tc_commit(drain);
      const uint32_t addr = ptx::smem_addr(drain);
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(addr, 0)) {
        if (ptx::globaltimer() - t0 > kTimeoutNs) { atomicOr(&g_device_error, kErrDrain); break; }
      }
    }
  } else if (warp == 2) {
    // --------------------------------------------------------- scale loader
    if (PROMOTE) {
      uint32_t ks = 0;
      bool ok = true;
      const int nb_first_stride = p.KB;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
        const int m0 = mt * kBM, n0 = nt * BN;
        for (int kb = 0; kb < KB; ++kb, ++ks) {
          const uint32_t slot = ks % kScaleSlots, sph = (ks / kScaleSlots) & 1;
          bool w = wait_bar(&sempty[slot], sph ^ 1, abort_flag, kErrScales);
          if (!__all_sync(0xFFFFFFFFu, w)) { ok = false; break; }
          float* dst = sScale + slot * L::kScaleFloats;
#pragma unroll
          for (int i = 0; i < kBM / 32; ++i) {
            const int r = lane + 32 * i, m = m0 + r;
            dst[r] = (m < p.M) ? __ldg(p.sa + (size_t)kb * p.M + m) : 0.0f;
          }
          float* dstb = dst + kBM;
          if (B_TILE) {
#pragma unroll
            for (int i = 0; i < BN / 32; ++i) {
              const int cidx = lane + 32 * i, n = n0 + cidx;
              dstb[cidx] = (n < p.N) ? __ldg(p.sb + (size_t)kb * p.N + n) : 0.0f;
            }
          } else if (lane < 4) {
            const int nb = n0 / 128 + lane;
            dstb[lane] = (nb * 128 < p.N) ? __ldg(p.sb + (size_t)nb * nb_first_stride + kb) : 0.0f;
          }
          ptx::mbar_arrive(&sfull[slot]);
        }
      }
    }
  } else if (warp >= kFirstPromoWarp) {
    // ------------------------------------------------- promotion + epilogue
    const int w = warp - kFirstPromoWarp;
    const int lg = warp & 3;       // TMEM lane group this warp may access
    const int ch = w >> 2;         // column half
    const int row = lg * 32 + lane;
    const int col0 = ch * kHalf;
    const uint32_t t_lane = (uint32_t)(lg * 32) << 16;
    uint32_t kt = 0, ks = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int m0 = mt * kBM, n0 = nt * BN;
      float acc[kHalf];
#pragma unroll
      for (int j = 0; j < kHalf; ++j) acc[j] = 0.0f;

      if (PROMOTE) {
        for (int kb = 0; kb < KB; ++kb, ++kt, ++ks) {
          const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
          const uint32_t slot = ks % kScaleSlots, sph = (ks / kScaleSlots) & 1;
          bool w1 = wait_bar(&sfull[slot], sph, abort_flag, kErrPromo);
          bool w2 = w1 && wait_bar(&tfull[buf], tph, abort_flag, kErrPromo);
          if (!__all_sync(0xFFFFFFFFu, w2)) { ok = false; break; }
          ptx::tc_fence_after();
          const float* sc = sScale + slot * L::kScaleFloats;
          const float sa_r = sc[row];
          const float* scb = sc + kBM;
          const uint32_t tbase = tmem_base + t_lane + buf * BN + col0;
#pragma unroll
          for (int c0 = 0; c0 < kChunks; c0 += kChunksPerRound) {
            uint32_t v[kChunksPerRound][32];
#pragma unroll
            for (int cc = 0; cc < kChunksPerRound; ++cc)
              ptx::tmem_ld_32x32b_x32(tbase + (c0 + cc) * 32, v[cc]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < kChunksPerRound; ++cc) ptx::reg_barrier(v[cc]);
            if (c0 + kChunksPerRound >= kChunks) {
              // every TMEM read of this buffer is done: hand it back
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&tempty[buf]);
            }
#pragma unroll
            for (int cc = 0; cc < kChunksPerRound; ++cc) {
              const int cbase = col0 + (c0 + cc) * 32;
              if (B_TILE) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const float f = __fmul_rn(sa_r, scb[cbase + j]);
                  acc[(c0 + cc) * 32 + j] =
                      __fmaf_rn(__uint_as_float(v[cc][j]), f, acc[(c0 + cc) * 32 + j]);
                }
              } else {
                const int nbi = (n0 + cbase) / 128 - n0 / 128;
                const float f = __fmul_rn(sa_r, scb[nbi]);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  acc[(c0 + cc) * 32 + j] =
                      __fmaf_rn(__uint_as_float(v[cc][j]), f, acc[(c0 + cc) * 32 + j]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sempty[slot]);
        }
      } else {
        const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
        bool w2 = wait_bar(&tfull[buf], tph, abort_flag, kErrPromo);
        if (!__all_sync(0xFFFFFFFFu, w2)) { ok = false; break; }
        ptx::tc_fence_after();
        const int m = m0 + row;
        const float sa_r = (m < p.M) ? __ldg(p.sa + m) : 0.0f;  // K-group 0
        const uint32_t tbase = tmem_base + t_lane + buf * BN + col0;
#pragma unroll
        for (int c0 = 0; c0 < kChunks; c0 += kChunksPerRound) {
          uint32_t v[kChunksPerRound][32];
#pragma unroll
          for (int cc = 0; cc < kChunksPerRound; ++cc)
            ptx::tmem_ld_32x32b_x32(tbase + (c0 + cc) * 32, v[cc]);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < kChunksPerRound; ++cc) ptx::reg_barrier(v[cc]);
#pragma unroll
          for (int cc = 0; cc < kChunksPerRound; ++cc) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = n0 + col0 + (c0 + cc) * 32 + j;
              float sbv = 0.0f;
              if (n < p.N) sbv = B_TILE ? __ldg(p.sb + n) : __ldg(p.sb + (size_t)(n / 128) * p.KB);
              acc[(c0 + cc) * 32 + j] =
                  __fmul_rn(__uint_as_float(v[cc][j]), __fmul_rn(sa_r, sbv));
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty[buf]);
        ++kt;
      }
      if (!ok) break;

      // ---- epilogue: registers -> global (bf16 RNE or fp32)
      const int m = m0 + row;
      if (m < p.M) {
        if (OUT_BF16) {
          __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(p.c) + (size_t)m * p.N;
#pragma unroll
          for (int j = 0; j < kHalf; j += 8) {
            const int n = n0 + col0 + j;
            if (n < p.N) {
              uint4 o;
              __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[j], acc[j + 1]);
              __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[j + 2], acc[j + 3]);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[j + 4], acc[j + 5]);
              __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[j + 6], acc[j + 7]);
              o.x = *reinterpret_cast<uint32_t*>(&b0);
              o.y = *reinterpret_cast<uint32_t*>(&b1);
              o.z = *reinterpret_cast<uint32_t*>(&b2);
              o.w = *reinterpret_cast<uint32_t*>(&b3);
              *reinterpret_cast<uint4*>(crow + n) = o;
            }
          }
        } else {
          float* crow = static_cast<float*>(p.c) + (size_t)m * p.N;
#pragma unroll
          for (int j = 0; j < kHalf; j += 4) {
            const int n = n0 + col0 + j;
            if (n < p.N)
              *reinterpret_cast<float4*>(crow + n) =
                  make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
          }
        }
      }
    }
  }

  // ---- teardown: all roles done (or aborted); free TMEM
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Row-major uint8 matrix [rows][cols] (cols contiguous), box of box_rows x
// 128 bytes with the 128-byte swizzle; out-of-range rows read as zero.
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms_current_device() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int BN, int STAGES, int TBUF, bool PROMOTE, bool OUT_BF16, bool B_TILE>
cudaError_t launch_variant(const GemmArgs& g, cudaStream_t stream) {
  using L = Smem<BN, STAGES, TBUF>;
  auto kern = gemm_kernel<BN, STAGES, TBUF, PROMOTE, OUT_BF16, B_TILE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, g.a, g.M, g.K, kBM) || !make_tmap(&tb, g.b, g.N, g.K, BN))
    return cudaErrorInvalidValue;
  Params p;
  p.sa = g.sa;
  p.sb = g.sb;
  p.c = g.c;
  p.M = (int)g.M;
  p.N = (int)g.N;
  p.K = (int)g.K;
  p.KB = (int)(g.K / kBK);
  p.num_m_tiles = (int)((g.M + kBM - 1) / kBM);
  const int num_n_tiles = (int)((g.N + BN - 1) / BN);
  p.num_tiles = p.num_m_tiles * num_n_tiles;
  p.skip_iter = g.skip_iter;
  int grid = num_sms_current_device();
  if (grid > p.num_tiles) grid = p.num_tiles;
  kern<<<grid, kThreads, L::kAlloc, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

template <bool PROMOTE, bool OUT_BF16, bool B_TILE>
cudaError_t launch_bn(const GemmArgs& g, cudaStream_t stream) {
  return launch_variant<128, 6, 4, PROMOTE, OUT_BF16, B_TILE>(g, stream);
}

template <bool PROMOTE, bool OUT_BF16>
cudaError_t launch_bt(const GemmArgs& g, cudaStream_t stream) {
  return g.b_tile ? launch_bn<PROMOTE, OUT_BF16, true>(g, stream)
                  : launch_bn<PROMOTE, OUT_BF16, false>(g, stream);
}

template <bool PROMOTE>
cudaError_t launch_out(const GemmArgs& g, cudaStream_t stream) {
  return g.out_bf16 ? launch_bt<PROMOTE, true>(g, stream) : launch_bt<PROMOTE, false>(g, stream);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  return g.promote ? launch_out<true>(g, stream) : launch_out<false>(g, stream);
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int* word) {
  *word = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = v;
  return cudaSuccess;
}

}  // namespace fp8bs
