// quant.cu -- the memory-bound quantizer kernels of libfp8bs:
//   Q1  1x128 activation tiles                         (page P1, para 3)
//   Q1T the same tiles laid 128x1, written transposed  (page P1, para 3)
//   Q2  128x128 weight blocks (+ transposed copy)      (page P1, para 3)
//   Q3  1x128 -> 128x1 re-tiling of cached FP8 codes   (page P1, para 3)
//
// All four read each input byte once and write each output byte once:
// 16-byte coalesced global loads, group max-abs by integer max on the sign-
// stripped bit patterns (monotone in |x| for non-NaN values; NaN patterns
// sort above Inf, so one compare also detects "group holds Inf/NaN"), and
// hardware E4M3x2 packing.  Groups that hold Inf/NaN, or whose scale is zero
// or tiny, take the general per-element path with an exact division; all
// others use the reciprocal-plus-correction quotient of fp8_common.cuh.
#include "fp8_common.cuh"
#include "launch.h"

namespace fp8bs {

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kBf16Inf = 0x7F80u;
constexpr uint32_t kF32Inf = 0x7F800000u;

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t mag2_max(uint32_t acc, uint32_t w) {
  acc = max(acc, w & 0x7FFFu);
  return max(acc, (w >> 16) & 0x7FFFu);
}

// Magnitude with NaN patterns replaced by 0 (NaN is ignored by amax).
__device__ __forceinline__ uint32_t mag_no_nan(uint32_t m, uint32_t inf) {
  return m > inf ? 0u : m;
}

__device__ __forceinline__ uint32_t mag2_max_no_nan(uint32_t acc, uint32_t w) {
  acc = max(acc, mag_no_nan(w & 0x7FFFu, kBf16Inf));
  return max(acc, mag_no_nan((w >> 16) & 0x7FFFu, kBf16Inf));
}

// Four bf16 pairs (one 16-byte vector) -> eight codes in two words.
struct GroupScale {
  float s, r;
  bool fast;
};

__device__ __forceinline__ GroupScale make_scale(uint32_t mag_bf16_no_nan, bool special) {
  GroupScale g;
  g.s = group_scale(__uint_as_float(mag_bf16_no_nan << 16));
  g.fast = !special && g.s >= kFastScaleMin;
  g.r = g.fast ? __frcp_rn(g.s) : 0.0f;
  return g;
}

__device__ __forceinline__ uint32_t codes_bf16x2(uint32_t w, const GroupScale& g) {
  float a = bf16_lo(w), b = bf16_hi(w);
  if (g.fast) return e4m3x2(quotient_1step(a, g.s, g.r), quotient_1step(b, g.s, g.r));
  return e4m3x2_nan(quotient_general(a, g.s), quotient_general(b, g.s));
}

__device__ __forceinline__ uint2 codes_bf16x8(uint4 v, const GroupScale& g) {
  uint2 o;
  o.x = codes_bf16x2(v.x, g) | (codes_bf16x2(v.y, g) << 16);
  o.y = codes_bf16x2(v.z, g) | (codes_bf16x2(v.w, g) << 16);
  return o;
}

// ---------------------------------------------------------------------------
// Q1: 1x128 tiles.  CTA = 256 threads = 16 half-warps; a half-warp owns one
// 128-element group (16 lanes x 8 bf16) of 4 rows; CTA tile 64 rows x one
// K-group.  grid = (ceil(M/64), K/128).
// ---------------------------------------------------------------------------
constexpr int kQ1Rows = 64;

__global__ void __launch_bounds__(256) quant_act_1x128_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t K, uint8_t* __restrict__ q,
    float* __restrict__ s) {
  const int64_t kb = blockIdx.y;
  const int hw = threadIdx.x >> 4;
  const int l16 = threadIdx.x & 15;
  const int64_t row0 = (int64_t)blockIdx.x * kQ1Rows + hw;
  const int64_t col = kb * kGroup + l16 * 8;

  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int64_t r = row0 + 16 * i;
    v[i] = (r < M) ? ld_stream_v4(x + r * K + col) : make_uint4(0, 0, 0, 0);
  }
  uint32_t mx[4];
  bool special = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t m = 0;
    m = mag2_max(m, v[i].x); m = mag2_max(m, v[i].y);
    m = mag2_max(m, v[i].z); m = mag2_max(m, v[i].w);
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
    mx[i] = m;
    special |= (m >= kBf16Inf);
  }
  bool sp[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) sp[i] = mx[i] >= kBf16Inf;
  if (__any_sync(kFull, special)) {  // warp-uniform: every lane shuffles
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t m = 0;
      m = mag2_max_no_nan(m, v[i].x); m = mag2_max_no_nan(m, v[i].y);
      m = mag2_max_no_nan(m, v[i].z); m = mag2_max_no_nan(m, v[i].w);
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
      mx[i] = m;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int64_t r = row0 + 16 * i;
    if (r >= M) continue;
    GroupScale g = make_scale(mx[i], sp[i]);
    *reinterpret_cast<uint2*>(q + r * K + col) = codes_bf16x8(v[i], g);
    if (l16 == 0) s[kb * M + r] = g.s;
  }
}

// ---------------------------------------------------------------------------
// Q1T: 128x1 tiles (groups of 128 consecutive rows of one column), output
// transposed.  CTA tile = 128 rows x 128 columns staged in shared memory.
// Thread (cp, p): column pair cp (0..63), rows p*32..p*32+31; a warp reads
// 32 consecutive words of one row (conflict-free).  grid = (K/128, M/128).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_act_128x1_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t K, uint8_t* __restrict__ qT,
    float* __restrict__ sT) {
  __shared__ uint4 tile[128 * 16];  // row r, 16-byte segment g at [r * 16 + g]
  __shared__ uint32_t red[4][64];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kGroup;
  const int64_t mb = blockIdx.y;
  const int64_t m0 = mb * kGroup;

#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int idx = t + 256 * j;
    int row = idx >> 4, g = idx & 15;
    tile[idx] = ld_stream_v4(x + (m0 + row) * K + k0 + g * 8);
  }
  __syncthreads();

  const uint32_t* tw = reinterpret_cast<const uint32_t*>(tile);
  const int cp = (t & 31) + 32 * ((t >> 5) & 1);
  const int p = t >> 6;
  uint32_t mlo = 0, mhi = 0;
#pragma unroll 8
  for (int i = 0; i < 32; ++i) {
    uint32_t w = tw[(p * 32 + i) * 64 + cp];
    mlo = max(mlo, w & 0x7FFFu);
    mhi = max(mhi, (w >> 16) & 0x7FFFu);
  }
  red[p][cp] = mlo | (mhi << 16);
  __syncthreads();
  mlo = 0; mhi = 0;
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    uint32_t w = red[pp][cp];
    mlo = max(mlo, w & 0xFFFFu);
    mhi = max(mhi, w >> 16);
  }
  const bool sp_lo = mlo >= kBf16Inf, sp_hi = mhi >= kBf16Inf;
  if (sp_lo || sp_hi) {  // rare: recount this column pair without NaN
    uint32_t a = 0, b = 0;
    for (int r = 0; r < 128; ++r) {
      uint32_t w = tw[r * 64 + cp];
      a = max(a, mag_no_nan(w & 0x7FFFu, kBf16Inf));
      b = max(b, mag_no_nan((w >> 16) & 0x7FFFu, kBf16Inf));
    }
    mlo = a; mhi = b;
  }
  const GroupScale glo = make_scale(mlo, sp_lo);
  const GroupScale ghi = make_scale(mhi, sp_hi);

  uint32_t olo[8], ohi[8];
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    uint32_t w0 = tw[(p * 32 + i) * 64 + cp];
    uint32_t w1 = tw[(p * 32 + i + 1) * 64 + cp];
    // pack (row i, row i+1) of each column: low column from the low halves
    uint32_t lo_pair = (w0 & 0xFFFFu) | (w1 << 16);
    uint32_t hi_pair = (w0 >> 16) | (w1 & 0xFFFF0000u);
    uint32_t clo = codes_bf16x2(lo_pair, glo);
    uint32_t chi = codes_bf16x2(hi_pair, ghi);
    if ((i & 2) == 0) {
      olo[i >> 2] = clo;
      ohi[i >> 2] = chi;
    } else {
      olo[i >> 2] |= clo << 16;
      ohi[i >> 2] |= chi << 16;
    }
  }
  uint8_t* dlo = qT + (k0 + 2 * cp) * M + m0 + p * 32;
  uint8_t* dhi = dlo + M;
  reinterpret_cast<uint4*>(dlo)[0] = make_uint4(olo[0], olo[1], olo[2], olo[3]);
  reinterpret_cast<uint4*>(dlo)[1] = make_uint4(olo[4], olo[5], olo[6], olo[7]);
  reinterpret_cast<uint4*>(dhi)[0] = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
  reinterpret_cast<uint4*>(dhi)[1] = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
  if (p == 0)
    *reinterpret_cast<float2*>(sT + mb * K + k0 + 2 * cp) = make_float2(glo.s, ghi.s);
}

// ---------------------------------------------------------------------------
// Q2: one CTA per 128x128 weight block.  Each thread holds 64 elements
// (8 x 16 bytes) in registers; the block max goes through shared memory.
// The optional transposed copy is staged as a row-major code tile in shared
// memory and read back column-wise (a warp reads 32 consecutive bytes).
// grid = (K/128, N/128).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_weight_128x128_kernel(
    const uint16_t* __restrict__ w, int64_t N, int64_t K, uint8_t* __restrict__ q,
    float* __restrict__ s, uint8_t* __restrict__ qT, float* __restrict__ sT) {
  __shared__ uint2 ctile[128 * 16];  // codes, row n, 8-byte segment g at [n * 16 + g]
  __shared__ uint32_t red[2][8];
  const int t = threadIdx.x;
  const int64_t kb = blockIdx.x, nb = blockIdx.y;
  const int64_t KB = K / kGroup, NB = N / kGroup;
  const int64_t n0 = nb * kGroup, k0 = kb * kGroup;

  uint4 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int idx = t + 256 * j;
    v[j] = ld_stream_v4(w + (n0 + (idx >> 4)) * K + k0 + (idx & 15) * 8);
  }
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    m = mag2_max(m, v[j].x); m = mag2_max(m, v[j].y);
    m = mag2_max(m, v[j].z); m = mag2_max(m, v[j].w);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
  if ((t & 31) == 0) red[0][t >> 5] = m;
  __syncthreads();
  m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, red[0][i]);
  const bool special = m >= kBf16Inf;  // block-uniform
  if (special) {
    m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      m = mag2_max_no_nan(m, v[j].x); m = mag2_max_no_nan(m, v[j].y);
      m = mag2_max_no_nan(m, v[j].z); m = mag2_max_no_nan(m, v[j].w);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
    if ((t & 31) == 0) red[1][t >> 5] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max(m, red[1][i]);
  }
  const GroupScale g = make_scale(m, special);

#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int idx = t + 256 * j;
    uint2 c = codes_bf16x8(v[j], g);
    *reinterpret_cast<uint2*>(q + (n0 + (idx >> 4)) * K + k0 + (idx & 15) * 8) = c;
    if (qT) ctile[idx] = c;
  }
  if (t == 0) {
    s[nb * KB + kb] = g.s;
    if (sT) sT[kb * NB + nb] = g.s;
  }
  if (qT) {
    __syncthreads();
    const uint8_t* cb = reinterpret_cast<const uint8_t*>(ctile);
    const int k = t & 127, h = t >> 7;
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int n = h * 64 + 4 * i;
      o[i] = (uint32_t)cb[n * 128 + k] | ((uint32_t)cb[(n + 1) * 128 + k] << 8) |
             ((uint32_t)cb[(n + 2) * 128 + k] << 16) | ((uint32_t)cb[(n + 3) * 128 + k] << 24);
    }
    uint4* d = reinterpret_cast<uint4*>(qT + (k0 + k) * N + n0 + h * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  }
}

// ---------------------------------------------------------------------------
// Q3: 1x128 -> 128x1.  CTA tile = 128 rows (one 128-token group) x 128
// columns (one K-group) of codes plus their 128 row scales, in shared
// memory.  Thread (cq, p): columns 4cq..4cq+3, rows p*16..p*16+15.
// x_hat = decode(code) * s_row (one RN multiply), then the column groups are
// quantized again and written transposed.  grid = (K/128, M/128).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dequant4(uint32_t w, float s, float (&o)[4]) {
  float2 a = e4m3x2_decode(w & 0xFFFFu);
  float2 b = e4m3x2_decode(w >> 16);
  o[0] = __fmul_rn(a.x, s); o[1] = __fmul_rn(a.y, s);
  o[2] = __fmul_rn(b.x, s); o[3] = __fmul_rn(b.y, s);
}

__global__ void __launch_bounds__(256) requant_1x128_to_128x1_kernel(
    const uint8_t* __restrict__ q, const float* __restrict__ s, int64_t M, int64_t K,
    uint8_t* __restrict__ qT, float* __restrict__ sT) {
  __shared__ uint4 tile[128 * 8];  // row r, 16-byte segment g at [r * 8 + g]
  __shared__ float srow[128];
  __shared__ uint32_t red[8][128];
  const int t = threadIdx.x;
  const int64_t kb = blockIdx.x, mb = blockIdx.y;
  const int64_t k0 = kb * kGroup, m0 = mb * kGroup;

#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int idx = t + 256 * j;
    tile[idx] = ld_stream_v4(q + (m0 + (idx >> 3)) * K + k0 + (idx & 7) * 16);
  }
  if (t < 128) srow[t] = s[kb * M + m0 + t];
  __syncthreads();

  const uint32_t* tw = reinterpret_cast<const uint32_t*>(tile);
  const int cq = t & 31, p = t >> 5;
  uint32_t mx[4] = {0, 0, 0, 0};
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int r = p * 16 + i;
    float xv[4];
    dequant4(tw[r * 32 + cq], srow[r], xv);
#pragma unroll
    for (int c = 0; c < 4; ++c) mx[c] = max(mx[c], __float_as_uint(xv[c]) & 0x7FFFFFFFu);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) red[p][4 * cq + c] = mx[c];
  __syncthreads();
  GroupScale g[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t m = 0;
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) m = max(m, red[pp][4 * cq + c]);
    const bool special = m >= kF32Inf;
    if (special) {  // rare: recount this column without NaN
      m = 0;
      for (int r = 0; r < 128; ++r) {
        float xv[4];
        dequant4(tw[r * 32 + cq], srow[r], xv);
        m = max(m, mag_no_nan(__float_as_uint(xv[c]) & 0x7FFFFFFFu, kF32Inf));
      }
    }
    g[c].s = group_scale(__uint_as_float(m));
    g[c].fast = !special && g[c].s >= kFastScaleMin;
    g[c].r = g[c].fast ? __frcp_rn(g[c].s) : 0.0f;
  }

  uint32_t o[4][4];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const int r = p * 16 + i;
    float x0[4], x1[4];
    dequant4(tw[r * 32 + cq], srow[r], x0);
    dequant4(tw[(r + 1) * 32 + cq], srow[r + 1], x1);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t code;
      if (g[c].fast)
        code = e4m3x2(quotient_2step(x0[c], g[c].s, g[c].r), quotient_2step(x1[c], g[c].s, g[c].r));
      else
        code = e4m3x2_nan(quotient_general(x0[c], g[c].s), quotient_general(x1[c], g[c].s));
      if ((i & 2) == 0)
        o[c][i >> 2] = code;
      else
        o[c][i >> 2] |= code << 16;
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(qT + (k0 + 4 * cq + c) * M + m0 + p * 16) =
        make_uint4(o[c][0], o[c][1], o[c][2], o[c][3]);
  if (p == 0)
    *reinterpret_cast<float4*>(sT + mb * K + k0 + 4 * cq) = make_float4(g[0].s, g[1].s, g[2].s, g[3].s);
}

}  // namespace

cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                   cudaStream_t stream) {
  dim3 grid((unsigned)((M + kQ1Rows - 1) / kQ1Rows), (unsigned)(K / kGroup));
  quant_act_1x128_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x), M, K, q, s);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, uint8_t* qT, float* sT,
                                   cudaStream_t stream) {
  dim3 grid((unsigned)(K / kGroup), (unsigned)(M / kGroup));
  quant_act_128x1_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x), M, K, qT, sT);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight_128x128(const void* w, int64_t N, int64_t K, uint8_t* q, float* s,
                                        uint8_t* qT, float* sT, cudaStream_t stream) {
  dim3 grid((unsigned)(K / kGroup), (unsigned)(N / kGroup));
  quant_weight_128x128_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(w), N, K, q,
                                                        s, qT, sT);
  return cudaGetLastError();
}

cudaError_t launch_requant_1x128_to_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                          uint8_t* qT, float* sT, cudaStream_t stream) {
  dim3 grid((unsigned)(K / kGroup), (unsigned)(M / kGroup));
  requant_1x128_to_128x1_kernel<<<grid, 256, 0, stream>>>(q, s, M, K, qT, sT);
  return cudaGetLastError();
}

}  // namespace fp8bs
