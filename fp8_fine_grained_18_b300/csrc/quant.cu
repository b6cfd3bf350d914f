// quant.cu -- the memory-bound quantizer kernels of libfp8bs:
//   Q1  1x128 activation tiles                         (page P1, para 3)
//   Q1T the same tiles laid 128x1, written transposed  (page P1, para 3)
//   Q2  128x128 weight blocks (+ transposed copy)      (page P1, para 3)
//   Q3  1x128 -> 128x1 re-tiling of cached FP8 codes   (page P1, para 3)
//   Q12 Q1 of an activation and Q2 of a weight in one launch
//   dual: Q1 and Q1T of one tensor from one read        (page P2, para 1)
//   Q1E5 / E5M6 re-tiling: the E5M6 cache of the re-tiled activations
//                                                       (page P1, para 3)
//   per-tensor baseline: one scale for the whole tensor (page P1, para 4;
//                                                        page P3, para 4)
//
// Q1 and Q2 are one streaming scheme: a persistent CTA per SM whose producer
// warp moves input tiles into a ring of shared-memory stages with 2-D TMA
// copies (mbarrier full/empty, every wait bounded), while 16 consumer warps
// turn each stage into codes and scales and store them.  Where a tile's
// threads must exchange group maxima, the consumers form teams (two of 8
// warps, or four of 4 for the E4M3 re-tiling) that work on alternate tiles,
// so one team's barrier waits overlap the others' work.  Tiles are ordered with the K-group fastest, so the CTAs
// running at one time read one contiguous band of the input.  Q12, Q1E5 and
// the transposing ops (Q1T and the dual quantizer as Q1TS, Q3 and the E5M6
// re-tiling as Q3S) are further ops of the same scheme: a team stages its
// transposed codes in a 128-byte-swizzled shared-memory tile that one thread
// writes out with a tensor store (and the scales with a bulk copy).  Each
// input byte is read from HBM once and each output byte written once.
//
// Group max-abs is an integer max on the sign-stripped bit patterns
// (monotone in |x| for non-NaN values; NaN patterns sort above Inf, so one
// compare also detects "group holds Inf/NaN"); only a tile that holds a NaN
// recomputes its maxima with NaN excluded.  Codes are packed two at a time
// by the hardware E4M3x2 converter.  Groups that hold Inf/NaN, or whose scale
// is zero or tiny, take the general per-element path with an exact division;
// all others use the reciprocal-plus-correction quotient of fp8_common.cuh.
#include <type_traits>

#include "fp8_common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace fp8bs {

__device__ unsigned int g_quant_error;  // set when a bounded wait gives up

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kBf16Inf = 0x7F80u;
constexpr uint32_t kF32Inf = 0x7F800000u;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;  // 512 consumer threads
constexpr int kThreads = kConsumers + 32;        // + one producer warp
constexpr uint64_t kTimeoutNs = 2000000000ull;   // 2 s per wait

// Max-abs on bf16 pairs: each 16-bit half keeps its own maximum magnitude
// bit pattern (packed unsigned max).
__device__ __forceinline__ uint32_t mag_pair_max(uint32_t acc, uint32_t w) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}

// The same with NaN patterns replaced by 0 (NaN is ignored by amax).
__device__ __forceinline__ uint32_t mag_pair_max_no_nan(uint32_t acc, uint32_t w) {
  const uint32_t m = w & 0x7FFF7FFFu;
  const uint32_t lo = (m & 0xFFFFu) > kBf16Inf ? 0u : (m & 0xFFFFu);
  const uint32_t hi = (m >> 16) > kBf16Inf ? 0u : (m >> 16);
  return __vmaxu2(acc, lo | (hi << 16));
}

__device__ __forceinline__ uint32_t halves_max(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }

__device__ __forceinline__ bool pair_has_nan(uint32_t m) {
  return (m & 0xFFFFu) > kBf16Inf || (m >> 16) > kBf16Inf;
}

// Four bf16 (two words, element 0 in the low half of wa) -> four codes,
// element 0 in byte 0.  The fast path converts the negated quotients and
// flips the four sign bits at once.
__device__ __forceinline__ uint32_t codes_bf16x4(uint32_t wa, uint32_t wb, const GroupScale& g) {
  const float2 xa = make_float2(bf16_lo(wa), bf16_hi(wa));
  const float2 xb = make_float2(bf16_lo(wb), bf16_hi(wb));
  if (g.fast) {
    const float2 qa = neg_quotient_1step_x2(xa, g.s, g.nr);
    const float2 qb = neg_quotient_1step_x2(xb, g.s, g.nr);
    return (e4m3x2(qa.x, qa.y) | (e4m3x2(qb.x, qb.y) << 16)) ^ 0x80808080u;
  }
  return e4m3x2_nan(quotient_general(xa.x, g.s), quotient_general(xa.y, g.s)) |
         (e4m3x2_nan(quotient_general(xb.x, g.s), quotient_general(xb.y, g.s)) << 16);
}

// Eight bf16 (one 16-byte vector) -> eight codes in two words.
__device__ __forceinline__ uint2 codes_bf16x8(uint4 v, const GroupScale& g) {
  return make_uint2(codes_bf16x4(v.x, v.y, g), codes_bf16x4(v.z, v.w, g));
}

// codes_bf16x4 for a group known to take the fast path, with the packed
// operands s2 = (s, s) and nr2 = (-1/s, -1/s) already formed: the same
// one-step quotient as neg_quotient_1step_x2.
__device__ __forceinline__ uint32_t codes_bf16x4_fast(uint32_t wa, uint32_t wb, float2 s2,
                                                      float2 nr2) {
  auto quot = [&](float2 x) {
    const float2 q0 = ptx::mul2_rn(x, nr2);
    return ptx::fma2_rn(ptx::fma2_rn(q0, s2, x), nr2, q0);
  };
  const float2 qa = quot(make_float2(bf16_lo(wa), bf16_hi(wa)));
  const float2 qb = quot(make_float2(bf16_lo(wb), bf16_hi(wb)));
  return (e4m3x2(qa.x, qa.y) | (e4m3x2(qb.x, qb.y) << 16)) ^ 0x80808080u;
}

__device__ __forceinline__ GroupScale shfl_scale(const GroupScale& g, int src) {
  GroupScale o;
  o.s = __shfl_sync(kFull, g.s, src);
  o.nr = __shfl_sync(kFull, g.nr, src);
  o.fast = __shfl_sync(kFull, (int)g.fast, src) != 0;
  return o;
}

// Bounded wait: false when it expired (the error word and the CTA's abort
// flag get set) or another warp already aborted.
__device__ __forceinline__ bool wait_q(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const uint32_t addr = ptx::smem_addr(bar);
#pragma unroll 1
  for (int i = 0; i < 128; ++i)
    if (ptx::mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(addr, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      atomicOr(&g_quant_error, 1u);
      return false;
    }
  }
}

// Consumer warp `warp` is done reading a stage.
__device__ __forceinline__ void release_stage(uint64_t* empty, int lane) {
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(empty);
}

// The consumer warps that work on one tile together.
struct Team {
  int tid;           // thread index within the team
  int warp;          // warp index within the team
  int lane;
  uint32_t bar;      // the team's named barrier
  uint32_t threads;  // threads in the team
  uint8_t* scratch;  // the team's shared-memory scratch
  uint64_t* empty;   // empty barrier of the stage being consumed
};

// 16 bytes into row k, chunk c of a 128 x 128 staging tile (128-byte swizzle).
__device__ __forceinline__ void stage_chunk(uint8_t* st, int k, int c, uint4 v) {
  *reinterpret_cast<uint4*>(st + k * 128 + ((c ^ (k & 7)) << 4)) = v;
}

// The team's staging buffer is free again once the previous tile's bulk
// stores (issued by the team's thread 0) have read it.
__device__ __forceinline__ void team_stage_wait(const Team& tm) {
  if (tm.tid == 0) ptx::bulk_wait_read_all();
}

// Store the staged tile: codes to (x = m0, y = k0) of the transposed output,
// and 128 scales to sT_row.  Called by every team thread after its staging
// writes.
__device__ __forceinline__ void team_stage_store(const Team& tm, const CUtensorMap* map_out,
                                                 const uint8_t* st, const float* st_scales,
                                                 int m0, int k0, float* sT_row) {
  ptx::fence_proxy_async_smem();
  ptx::named_barrier(tm.bar, tm.threads);
  if (tm.tid == 0) {
    ptx::tma_store_2d(map_out, st, m0, k0);
    ptx::bulk_store(sT_row, st_scales, 128 * 4);
    ptx::bulk_commit();
  }
}

// Q1's per-row maxima: half-warp rows h, h+32, h+64, h+96, eight bf16 of
// each per lane (v[i] for row i).  Returns in lane j (0..3) of the half-warp
// row j's NaN-free max magnitude (mj) and its plain max (pj >= Inf flags a
// group with Inf or NaN), both as bf16 bit patterns.
__device__ __forceinline__ void q1_row_max(const uint4* v, int l16, uint32_t& mj, uint32_t& pj) {
  // per-row maxima, two rows packed per word, reduced over the half-warp
  uint32_t m01 = 0, m23 = 0;
  {
    uint32_t a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      a[i] = halves_max(mag_pair_max(mag_pair_max(mag_pair_max(mag_pair_max(0u, v[i].x), v[i].y),
                                                  v[i].z),
                                     v[i].w));
    m01 = a[0] | (a[1] << 16);
    m23 = a[2] | (a[3] << 16);
  }
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
    m01 = __vmaxu2(m01, __shfl_xor_sync(kFull, m01, off));
    m23 = __vmaxu2(m23, __shfl_xor_sync(kFull, m23, off));
  }
  const uint32_t plain01 = m01, plain23 = m23;
  if (__any_sync(kFull, pair_has_nan(m01) || pair_has_nan(m23))) {  // recount without NaN
    uint32_t a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      a[i] = halves_max(mag_pair_max_no_nan(
          mag_pair_max_no_nan(mag_pair_max_no_nan(mag_pair_max_no_nan(0u, v[i].x), v[i].y),
                              v[i].z),
          v[i].w));
    m01 = a[0] | (a[1] << 16);
    m23 = a[2] | (a[3] << 16);
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
      m01 = __vmaxu2(m01, __shfl_xor_sync(kFull, m01, off));
      m23 = __vmaxu2(m23, __shfl_xor_sync(kFull, m23, off));
    }
  }
  const int j = l16 & 3;
  const uint32_t mw = j < 2 ? m01 : m23, pw = j < 2 ? plain01 : plain23;
  mj = (j & 1) ? (mw >> 16) : (mw & 0xFFFFu);
  pj = (j & 1) ? (pw >> 16) : (pw & 0xFFFFu);
}

// The same for groups of 8 lanes that own four rows, lane l8 holding two
// 8-element halves of each (v[2 i], v[2 i + 1] for row i): rows 0, 1 and
// 2, 3 reduce packed in one word each over the group's three shuffle
// levels; lane l8 gets row (l8 & 3)'s maxima.
__device__ __forceinline__ void q1_row_max8(const uint4 (&v)[8], int l8, uint32_t& mj,
                                            uint32_t& pj) {
  auto reduce = [&](bool no_nan, uint32_t& m01, uint32_t& m23) {
    uint32_t a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t ws[8] = {v[2 * i].x,     v[2 * i].y,     v[2 * i].z,     v[2 * i].w,
                              v[2 * i + 1].x, v[2 * i + 1].y, v[2 * i + 1].z, v[2 * i + 1].w};
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) m = no_nan ? mag_pair_max_no_nan(m, ws[k]) : mag_pair_max(m, ws[k]);
      a[i] = halves_max(m);
    }
    m01 = a[0] | (a[1] << 16);
    m23 = a[2] | (a[3] << 16);
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) {
      m01 = __vmaxu2(m01, __shfl_xor_sync(kFull, m01, off));
      m23 = __vmaxu2(m23, __shfl_xor_sync(kFull, m23, off));
    }
  };
  uint32_t m01, m23;
  reduce(false, m01, m23);
  const uint32_t p01 = m01, p23 = m23;
  if (__any_sync(kFull, pair_has_nan(m01) || pair_has_nan(m23))) reduce(true, m01, m23);
  const int j = l8 & 3;
  const uint32_t mw = j < 2 ? m01 : m23, pw = j < 2 ? p01 : p23;
  mj = (j & 1) ? (mw >> 16) : (mw & 0xFFFFu);
  pj = (j & 1) ? (pw >> 16) : (pw & 0xFFFFu);
}

// ---------------------------------------------------------------------------
// Q1: 1x128 tiles.  Tile = 128 rows x one K-group (TMA box 128 x 128 bf16,
// 32 KB).  Half-warp h (0..31) owns rows h, h + 32, h + 64, h + 96 of the
// tile, each lane 8 consecutive elements of each; lanes 0..3 of the
// half-warp compute the four groups' scales and share them by shuffle.
// ---------------------------------------------------------------------------
struct Q1 {
  static constexpr int kRows = 128;
  static constexpr int kStageBytes = kRows * 256;
  static constexpr int kStages = 4;
  static constexpr int kScratchBytes = 0;
  static constexpr uint32_t kTx = kStageBytes;
  static constexpr int kTeams = 1;
  static constexpr bool kBulkStores = false;
  struct Params {
    uint8_t* q;
    float* s;
    int M, K, KB, num_tiles;
    const float* unused;
  };
  __device__ static void issue(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile,
                               const Params& p) {
    ptx::tma_load_2d(dst, map, bar, (tile % p.KB) * kGroup, (tile / p.KB) * kRows);
  }
  // R rows per half-warp (4: all 16 consumer warps share a tile; a team of
  // 8 warps, in the fused activation + weight launch, takes consume_team8).
  template <int R = 4>
  __device__ static void consume(const uint8_t* stage, int tile, const Params& p,
                                 const Team& tm) {
    constexpr int kHalfWarps = kRows / R;
    const int kb = tile % p.KB, rt = tile / p.KB;
    const int lane = tm.lane;
    const int hw = tm.warp * 2 + (lane >> 4);
    const int l16 = lane & 15;
    const uint4* st = reinterpret_cast<const uint4*>(stage);
    uint4 v[R];
#pragma unroll
    for (int i = 0; i < R; ++i) v[i] = st[(hw + kHalfWarps * i) * 16 + l16];
    uint32_t mj[R / 4], pj[R / 4];
#pragma unroll
    for (int b = 0; b < R / 4; ++b) q1_row_max(v + 4 * b, l16, mj[b], pj[b]);
    release_stage(tm.empty, lane);
    const int64_t col = (int64_t)kb * kGroup + l16 * 8;
#pragma unroll
    for (int b = 0; b < R / 4; ++b) {
      // lane i (< 4) of the half-warp made row 4b + i's scale; -1/s is 0
      // off the fast path, and one vote takes the warp's rows down it
      const GroupScale mine = make_scale(mj[b], pj[b] >= kBf16Inf, true);
      const float nmine = mine.fast ? mine.nr : 0.0f;
      if (__all_sync(kFull, l16 >= 4 || mine.fast)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float si = __shfl_sync(kFull, mine.s, (lane & 16) + i);
          const float ni = __shfl_sync(kFull, nmine, (lane & 16) + i);
          const float2 s2 = make_float2(si, si), n2 = make_float2(ni, ni);
          const int64_t r = (int64_t)rt * kRows + hw + kHalfWarps * (4 * b + i);
          const uint4 x = v[4 * b + i];
          if (r < p.M) {
            *reinterpret_cast<uint2*>(p.q + r * p.K + col) =
                make_uint2(codes_bf16x4_fast(x.x, x.y, s2, n2), codes_bf16x4_fast(x.z, x.w, s2, n2));
            if (l16 == i) p.s[(int64_t)kb * p.M + r] = mine.s;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const GroupScale g = shfl_scale(mine, (lane & 16) + i);
          const int64_t r = (int64_t)rt * kRows + hw + kHalfWarps * (4 * b + i);
          if (r < p.M) {
            *reinterpret_cast<uint2*>(p.q + r * p.K + col) = codes_bf16x8(v[4 * b + i], g);
            if (l16 == i) p.s[(int64_t)kb * p.M + r] = mine.s;
          }
        }
      }
    }
  }
  // A team of 8 warps (the fused activation + weight launch): each group of
  // 8 lanes owns rows g8 + 32 i (i < 4) of the tile and lane l8 elements
  // 8 l8 .. 8 l8 + 7 and 64 + 8 l8 .. 64 + 8 l8 + 7 of each; lane i (< 4)
  // of the group makes row i's scale, one per lane (a half-warp per row
  // would give each scale-making lane two).
  __device__ static void consume_team8(const uint8_t* stage, int tile, const Params& p,
                                       const Team& tm) {
    const int kb = tile % p.KB, rt = tile / p.KB;
    const int lane = tm.lane;
    const int g8 = tm.warp * 4 + (lane >> 3), l8 = lane & 7, gbase = lane & ~7;
    const uint4* st = reinterpret_cast<const uint4*>(stage);
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = st[(g8 + 32 * i) * 16 + l8];
      v[2 * i + 1] = st[(g8 + 32 * i) * 16 + 8 + l8];
    }
    uint32_t mj, pj;
    q1_row_max8(v, l8, mj, pj);
    release_stage(tm.empty, lane);
    const int64_t col = (int64_t)kb * kGroup + l8 * 8;
    const GroupScale mine = make_scale(mj, pj >= kBf16Inf, true);
    const float nmine = mine.fast ? mine.nr : 0.0f;
    if (__all_sync(kFull, l8 >= 4 || mine.fast)) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float si = __shfl_sync(kFull, mine.s, gbase + i);
        const float ni = __shfl_sync(kFull, nmine, gbase + i);
        const float2 s2 = make_float2(si, si), n2 = make_float2(ni, ni);
        const int64_t r = (int64_t)rt * kRows + g8 + 32 * i;
        if (r < p.M) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 x = v[2 * i + h];
            *reinterpret_cast<uint2*>(p.q + r * p.K + col + 64 * h) =
                make_uint2(codes_bf16x4_fast(x.x, x.y, s2, n2), codes_bf16x4_fast(x.z, x.w, s2, n2));
          }
          if (l8 == i) p.s[(int64_t)kb * p.M + r] = mine.s;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const GroupScale g = shfl_scale(mine, gbase + i);
        const int64_t r = (int64_t)rt * kRows + g8 + 32 * i;
        if (r < p.M) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            *reinterpret_cast<uint2*>(p.q + r * p.K + col + 64 * h) = codes_bf16x8(v[2 * i + h], g);
          if (l8 == i) p.s[(int64_t)kb * p.M + r] = mine.s;
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Q1E5: the E5M6 cache of an activation that will be re-tiled for the
// weight gradient (page P1, paragraph 3), optionally with its E4M3 1x128
// codes for the forward GEMM from the same read.  Same tiles and thread
// layout as Q1; each lane writes its eight 12-bit codes as three words.
// ---------------------------------------------------------------------------

// Fast-path E5M6 code of a negated quotient q = -x/s with bit pattern ux
// (finite, |q| <= 65024; the code's sign is the complement of q's).  Normal
// range: round the FP32 pattern to 6 mantissa bits with ties to even by one
// integer addition (exponent and mantissa fields are adjacent, so a carry
// lands in the exponent), which also rebiases the exponent by 112 steps
// (7168 = 112 * 64, i.e. 7168 << 17 subtracted before the shift; the
// pattern is at least 113 << 23 there, so nothing wraps).  Below 2^-14 the
// multiple of 2^-20 comes from one fused multiply-add, |q| * 2^20 + 2^23,
// whose product is exact and whose sum rounds to nearest even at an ulp of 1.
__device__ __forceinline__ uint32_t e5m6_code_negq(uint32_t ux) {
  const uint32_t a = ux & 0x7FFFFFFFu;
  const uint32_t norm = (a + ((a >> 17) & 1u) + (0xFFFFu - (7168u << 17))) >> 17;
  const uint32_t sub = __float_as_uint(__fmaf_rn(__uint_as_float(a), 0x1.0p20f, 0x1.0p23f)) & 0x7Fu;
  return ((~ux >> 20) & 0x800u) | (a < 0x38800000u ? sub : norm);
}

struct Q1E5 {
  static constexpr int kRows = 128;
  static constexpr int kStageBytes = kRows * 256;
  static constexpr int kStages = 4;
  static constexpr int kScratchBytes = 0;
  static constexpr uint32_t kTx = kStageBytes;
  static constexpr int kTeams = 1;
  static constexpr bool kBulkStores = false;
  struct Params {
    uint8_t* e5;  // [M][3K/2]
    float* s5;    // [K/128][M]
    uint8_t* q;   // E4M3 [M][K] or null
    float* s;     // [K/128][M] or null
    int M, K, KB, num_tiles;
  };
  __device__ static void issue(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile,
                               const Params& p) {
    ptx::tma_load_2d(dst, map, bar, (tile % p.KB) * kGroup, (tile / p.KB) * kRows);
  }
  __device__ static void consume(const uint8_t* stage, int tile, const Params& p,
                                 const Team& tm) {
    const int kb = tile % p.KB, rt = tile / p.KB;
    const int lane = tm.lane;
    const int hw = tm.warp * 2 + (lane >> 4);
    const int l16 = lane & 15;
    const uint4* st = reinterpret_cast<const uint4*>(stage);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = st[(hw + 32 * i) * 16 + l16];
    uint32_t mj, pj;
    q1_row_max(v, l16, mj, pj);
    release_stage(tm.empty, lane);
    const GroupScale mine5 = make_scale(mj, pj >= kBf16Inf, true, kE5M6Max);
    const GroupScale mine8 = make_scale(mj, pj >= kBf16Inf, true);
    const int64_t col = (int64_t)kb * kGroup + l16 * 8;
    const int64_t row_bytes = (int64_t)p.K / 2 * 3;
    // one vote: when all four rows' groups of the warp take the fast
    // quotient for both formats, only s and -1/s are broadcast and no call
    // tests a flag
    if (__all_sync(kFull, l16 >= 4 || (mine5.fast && mine8.fast))) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int src = (lane & 16) + i;
        const float s5 = __shfl_sync(kFull, mine5.s, src);
        const float n5 = __shfl_sync(kFull, mine5.nr, src);
        const float2 s52 = make_float2(s5, s5), n52 = make_float2(n5, n5);
        const int64_t r = (int64_t)rt * kRows + hw + 32 * i;
        uint32_t c[8];
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x = make_float2(bf16_lo(w[k]), bf16_hi(w[k]));
          const float2 q0 = ptx::mul2_rn(x, n52);
          const float2 qn = ptx::fma2_rn(ptx::fma2_rn(q0, s52, x), n52, q0);
          const uint32_t ux = __float_as_uint(qn.x), uy = __float_as_uint(qn.y);
          c[2 * k] = e5m6_code_negq(ux);
          c[2 * k + 1] = e5m6_code_negq(uy);
        }
        if (p.q) {
          const float s8 = __shfl_sync(kFull, mine8.s, src);
          const float n8 = __shfl_sync(kFull, mine8.nr, src);
          const float2 s82 = make_float2(s8, s8), n82 = make_float2(n8, n8);
          if (r < p.M) {
            *reinterpret_cast<uint2*>(p.q + r * p.K + col) =
                make_uint2(codes_bf16x4_fast(v[i].x, v[i].y, s82, n82),
                           codes_bf16x4_fast(v[i].z, v[i].w, s82, n82));
            if (l16 == i) p.s[(int64_t)kb * p.M + r] = mine8.s;
          }
        }
        if (r < p.M) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(p.e5 + r * row_bytes + col / 2 * 3);
          const uint3 pk = e5m6_pack8(c);
          dst[0] = pk.x;
          dst[1] = pk.y;
          dst[2] = pk.z;
          if (l16 == i) p.s5[(int64_t)kb * p.M + r] = mine5.s;
        }
      }
      return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const GroupScale g5 = shfl_scale(mine5, (lane & 16) + i);
      const int64_t r = (int64_t)rt * kRows + hw + 32 * i;
      uint32_t c[8];
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      if (g5.fast) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 qn =
              neg_quotient_1step_x2(make_float2(bf16_lo(w[k]), bf16_hi(w[k])), g5.s, g5.nr);
          const uint32_t ux = __float_as_uint(qn.x), uy = __float_as_uint(qn.y);
          c[2 * k] = e5m6_code_negq(ux);
          c[2 * k + 1] = e5m6_code_negq(uy);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          c[2 * k] = e5m6_of(quotient_general(bf16_lo(w[k]), g5.s));
          c[2 * k + 1] = e5m6_of(quotient_general(bf16_hi(w[k]), g5.s));
        }
      }
      if (p.q) {
        const GroupScale g8 = shfl_scale(mine8, (lane & 16) + i);
        if (r < p.M) {
          *reinterpret_cast<uint2*>(p.q + r * p.K + col) = codes_bf16x8(v[i], g8);
          if (l16 == i) p.s[(int64_t)kb * p.M + r] = mine8.s;
        }
      }
      if (r < p.M) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.e5 + r * row_bytes + col / 2 * 3);
        const uint3 pk = e5m6_pack8(c);
        dst[0] = pk.x;
        dst[1] = pk.y;
        dst[2] = pk.z;
        if (l16 == i) p.s5[(int64_t)kb * p.M + r] = mine5.s;
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Q2: 128x128 weight blocks.  Tile = one block (TMA box 128 x 128 bf16,
// 32 KB), one team of 256 threads.  Thread t holds elements (row, 8-column
// segment) for idx = t + 256 j, row = idx / 16, segment = idx % 16; the
// block max goes through shared memory.  The transposed copy is staged as a
// code tile in the team's scratch and read back column-wise, 32 contiguous
// bytes per thread.
// ---------------------------------------------------------------------------
struct Q2 {
  static constexpr int kStageBytes = 128 * 256;
  static constexpr int kStages = 4;
  static constexpr int kTeamWarps = 8;
  // scratch: the transposed copy's staging tile (1024-byte aligned, first),
  // the block's code tile, the max reduction
  static constexpr int kOffCodes = 128 * 128;
  static constexpr int kOffRed = kOffCodes + 128 * 128;
  static constexpr int kScratchBytes = kOffRed + 2 * kTeamWarps * 4;
  static constexpr uint32_t kTx = kStageBytes;
  static constexpr int kTeams = 2;
  static constexpr bool kBulkStores = true;
  struct Params {
    CUtensorMap map_t;  // qT [K][N] bytes, 128 x 128 box, 128-byte swizzle (64-byte aligned)
    uint8_t* q;
    float* s;
    uint8_t* qT;  // null: no transposed copy
    float* sT;
    int N, K, KB, NB, num_tiles;
  };
  __device__ static void issue(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile,
                               const Params& p) {
    ptx::tma_load_2d(dst, map, bar, (tile % p.KB) * kGroup, (tile / p.KB) * kGroup);
  }
  __device__ static void consume(const uint8_t* stage, int tile, const Params& p,
                                 const Team& tm) {
    const int kb = tile % p.KB, nb = tile / p.KB;
    const int t = tm.tid;
    const uint4* st = reinterpret_cast<const uint4*>(stage);
    uint2* ctile = reinterpret_cast<uint2*>(tm.scratch + kOffCodes);
    uint32_t* red = reinterpret_cast<uint32_t*>(tm.scratch + kOffRed);
    uint4 v[8];
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = st[t + 256 * j];
      m2 = mag_pair_max(mag_pair_max(mag_pair_max(mag_pair_max(m2, v[j].x), v[j].y), v[j].z),
                        v[j].w);
    }
    release_stage(tm.empty, tm.lane);
    if (p.qT) team_stage_wait(tm);  // the staging tile is free again
    uint32_t m = halves_max(m2);
    const bool nan_here = m > kBf16Inf;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
    if (tm.lane == 0) red[tm.warp] = m;
    const bool any_nan = ptx::named_barrier_or(tm.bar, tm.threads, nan_here);
    uint32_t mp = 0;
#pragma unroll
    for (int i = 0; i < kTeamWarps; ++i) mp = max(mp, red[i]);
    uint32_t mn = mp;
    if (any_nan) {  // uniform: recount without NaN
      uint32_t a2 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        a2 = mag_pair_max_no_nan(
            mag_pair_max_no_nan(mag_pair_max_no_nan(mag_pair_max_no_nan(a2, v[j].x), v[j].y),
                                v[j].z),
            v[j].w);
      uint32_t a = halves_max(a2);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) a = max(a, __shfl_xor_sync(kFull, a, off));
      if (tm.lane == 0) red[kTeamWarps + tm.warp] = a;
      ptx::named_barrier(tm.bar, tm.threads);
      mn = 0;
#pragma unroll
      for (int i = 0; i < kTeamWarps; ++i) mn = max(mn, red[kTeamWarps + i]);
    }
    const GroupScale g = make_scale(mn, mp >= kBf16Inf, true);
    const int64_t n0 = (int64_t)nb * kGroup, k0 = (int64_t)kb * kGroup;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int idx = t + 256 * j;
      const uint2 cv = codes_bf16x8(v[j], g);
      *reinterpret_cast<uint2*>(p.q + (n0 + (idx >> 4)) * p.K + k0 + (idx & 15) * 8) = cv;
      if (p.qT) ctile[idx] = cv;
    }
    if (t == 0) {
      p.s[(int64_t)nb * p.KB + kb] = g.s;
      if (p.sT) p.sT[(int64_t)kb * p.NB + nb] = g.s;
    }
    if (p.qT) {
      // The transposed copy: thread (kq, chunk) reads words kq (codes
      // 4 kq .. 4 kq + 3) of rows 16 chunk .. 16 chunk + 15 of the code tile,
      // transposes the 16 x 4 bytes with byte permutes into output rows
      // 4 kq + c (16 codes each), and stages them for one tensor store.
      ptx::named_barrier(tm.bar, tm.threads);
      const uint32_t* cw = reinterpret_cast<const uint32_t*>(ctile);
      const int kq = t & 31, chunk = t >> 5;
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = cw[(16 * chunk + i) * 32 + kq];
      uint32_t o[4][4];  // o[c][j]: output row 4 kq + c, rows 4 j .. 4 j + 3 of the chunk
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t a = w[4 * j], b = w[4 * j + 1], c = w[4 * j + 2], d = w[4 * j + 3];
        const uint32_t ab01 = __byte_perm(a, b, 0x5140), cd01 = __byte_perm(c, d, 0x5140);
        const uint32_t ab23 = __byte_perm(a, b, 0x7362), cd23 = __byte_perm(c, d, 0x7362);
        o[0][j] = __byte_perm(ab01, cd01, 0x5410);
        o[1][j] = __byte_perm(ab01, cd01, 0x7632);
        o[2][j] = __byte_perm(ab23, cd23, 0x5410);
        o[3][j] = __byte_perm(ab23, cd23, 0x7632);
      }
      // lane kq writes row c' = (c + kq / 2) % 4 at step c (conflict-free)
      const int rot = (kq >> 1) & 3;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = (c + rot) & 3;
        uint4 d = make_uint4(o[0][0], o[0][1], o[0][2], o[0][3]);
        if (cc == 1) d = make_uint4(o[1][0], o[1][1], o[1][2], o[1][3]);
        if (cc == 2) d = make_uint4(o[2][0], o[2][1], o[2][2], o[2][3]);
        if (cc == 3) d = make_uint4(o[3][0], o[3][1], o[3][2], o[3][3]);
        stage_chunk(tm.scratch, 4 * kq + cc, chunk, d);
      }
      ptx::fence_proxy_async_smem();
      ptx::named_barrier(tm.bar, tm.threads);
      if (t == 0) {
        ptx::tma_store_2d(&p.map_t, tm.scratch, (int)n0, (int)k0);
        ptx::bulk_commit();
      }
    }
  }
};

template <class Op>
struct StreamSmem {
  // Each team's scratch comes first, 1024-byte aligned (a bulk tensor store
  // with the 128-byte swizzle reads its staging buffer from there), then the
  // ring of input stages, then the barriers.
  static constexpr int kScratchPerTeam = ((Op::kScratchBytes + 1023) / 1024) * 1024;
  static constexpr int kOffScratch = 0;
  static constexpr int kOffRing = Op::kTeams * kScratchPerTeam;
  static constexpr int kRing = Op::kStages * Op::kStageBytes;
  static constexpr int kOffBars = kOffRing + kRing;
  static constexpr int kBytes = kOffBars + 2 * Op::kStages * 8 + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
  static_assert(Op::kStageBytes % 128 == 0, "stage alignment");
  static_assert(Op::kStages <= 32, "stage mask");
  static_assert(kAlloc <= 232448, "shared memory");
  // team t consumes the tiles at ring positions t, t + kTeams, ..., so each
  // stage belongs to one team
  static_assert(Op::kStages % Op::kTeams == 0, "stages per team");
  static_assert(kConsumerWarps % Op::kTeams == 0, "warps per team");
};

// The streaming kernel: warp kConsumerWarps is the producer, warps
// 0..kConsumerWarps-1 consume, in Op::kTeams teams.  CTA i handles tiles
// i, i + grid, ...; its j-th tile goes to team j mod kTeams.
template <class Op>
__global__ void __launch_bounds__(kThreads, 1)
    stream_kernel(const __grid_constant__ CUtensorMap map,
                  const __grid_constant__ typename Op::Params p) {
  using L = StreamSmem<Op>;
  constexpr int S = Op::kStages;
  constexpr int kTeamWarps = kConsumerWarps / Op::kTeams;
  // A programmatic dependent (the GEMM) may start on SMs this grid leaves;
  // it waits for this grid's completion before reading what it wrote.
  asm volatile("griddepcontrol.launch_dependents;");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + L::kOffRing;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
  uint64_t* empty = full + S;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], kTeamWarps);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&map);
      uint32_t it = 0, issued = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
        const uint32_t s = it % S, ph = (it / S) & 1;
        if (!wait_q(&empty[s], ph ^ 1, abort_flag)) break;
        ptx::mbar_arrive_expect_tx(&full[s], Op::kTx);
        Op::issue(&map, ring + s * Op::kStageBytes, &full[s], tile, p);
        issued |= 1u << s;
      }
      // Drain: the last copy issued into each stage has landed before the
      // CTA may exit (only the last phase of a stage can be in flight).
      for (uint32_t s = 0; s < S; ++s) {
        if (!((issued >> s) & 1u)) continue;
        const uint32_t li = (it - 1) - (((it - 1) % S + S - s) % S);
        const uint32_t addr = ptx::smem_addr(&full[s]);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(addr, (li / S) & 1)) {
          if (ptx::globaltimer() - t0 > kTimeoutNs) {
            atomicOr(&g_quant_error, 2u);
            break;
          }
        }
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    const int team = warp / kTeamWarps;
    Team tm;
    tm.warp = warp % kTeamWarps;
    tm.lane = lane;
    tm.tid = tm.warp * 32 + lane;
    tm.bar = 1 + team;
    tm.threads = 32 * kTeamWarps;
    tm.scratch = smem + L::kOffScratch + team * L::kScratchPerTeam;
    uint32_t it = team;
    for (int tile = blockIdx.x + team * gridDim.x; tile < p.num_tiles;
         tile += Op::kTeams * gridDim.x, it += Op::kTeams) {
      const uint32_t s = it % S, ph = (it / S) & 1;
      const bool ok = wait_q(&full[s], ph, abort_flag);
      // A team whose threads synchronize with each other decides together
      // (this barrier also separates the previous tile's use of the team's
      // scratch from this one's); single warps decide alone.
      if (kTeamWarps > 1 && Op::kTeams > 1) {
        if (ptx::named_barrier_or(tm.bar, tm.threads, !ok)) break;
      } else {
        if (!__all_sync(kFull, ok)) break;
      }
      tm.empty = &empty[s];
      Op::consume(ring + s * Op::kStageBytes, tile, p, tm);
    }
    // a team's bulk stores read its staging buffer and write the output:
    // both are complete before the CTA exits
    if constexpr (Op::kBulkStores) {
      if (tm.tid == 0) ptx::bulk_wait_all();
    }
  }
}


__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Q12: both operands of the forward GEMM in one launch -- an activation's
// 1x128 tiles (tiles 0 .. t1-1, through the kernel's tensor map) and a
// weight's 128x128 blocks (tiles t1 .., through map_w).  Both tile kinds are
// 128 x 128 bf16 (32 KB); two teams of 8 warps take alternate tiles, so a
// team quantizes an activation tile with 8 rows per half-warp.  One launch
// pays the launch, ramp and tail once for the two tensors.
// ---------------------------------------------------------------------------
struct Q12 {
  static constexpr int kStageBytes = 128 * 256;
  static constexpr int kStages = 4;
  static constexpr int kScratchBytes = Q2::kScratchBytes;
  static constexpr uint32_t kTx = kStageBytes;
  static constexpr int kTeams = 2;
  static constexpr bool kBulkStores = true;
  static_assert(Q1::kStageBytes == kStageBytes && Q2::kStageBytes == kStageBytes, "tile size");
  static_assert(Q2::kTeams == kTeams && Q2::kTeamWarps == kConsumerWarps / kTeams, "teams");
  struct Params {
    CUtensorMap map_w;  // 64-byte aligned: first member
    Q1::Params a;
    Q2::Params w;
    int t1, num_tiles;
  };
  __device__ static void issue(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile,
                               const Params& p) {
    if (tile < p.t1)
      Q1::issue(map, dst, bar, tile, p.a);
    else
      Q2::issue(&p.map_w, dst, bar, tile - p.t1, p.w);
  }
  __device__ static void consume(const uint8_t* stage, int tile, const Params& p,
                                 const Team& tm) {
    if (tile < p.t1)
      Q1::consume_team8(stage, tile, p.a, tm);
    else
      Q2::consume(stage, tile - p.t1, p.w, tm);
  }
};

// ---------------------------------------------------------------------------
// Per-tensor baseline: one scale for the whole tensor, from its max-abs
// mapped to the FP8 maximum (the standard practice that the fine-grained
// tiles replace, kept to measure what they gain).  Three stream-ordered
// launches with no scratch memory: pass 1 folds the NaN-free bf16 magnitudes
// into the caller's scale word with one atomicMax per CTA (the FP32 bits of
// non-negative values order like unsigned integers, and a bf16 magnitude
// shifted left by 16 is its FP32 bit pattern); pass 2 quantizes with
// s = fl32(amax / 448) and writes the optional broadcast copy of s; pass 3,
// one thread, replaces the amax in the scale word by s.
// ---------------------------------------------------------------------------
constexpr int kPtThreads = 512;
constexpr int kPtCtasPerSm = 4;  // 2048 threads per SM

// The two bf16 magnitudes of a word, NaN lanes set to zero.
__device__ __forceinline__ uint32_t mag_no_nan2(uint32_t w) {
  const uint32_t mag = w & 0x7FFF7FFFu;
  return mag & ~__vcmpgtu2(mag, 0x7F807F80u);
}

__device__ __forceinline__ uint32_t mag_max8(const uint4& v) {
  return __vmaxu2(__vmaxu2(mag_no_nan2(v.x), mag_no_nan2(v.y)),
                  __vmaxu2(mag_no_nan2(v.z), mag_no_nan2(v.w)));
}

__device__ __forceinline__ bool has_nan8(const uint4& v) {
  const uint32_t inf2 = 0x7F807F80u;
  return (__vcmpgtu2(v.x & 0x7FFF7FFFu, inf2) | __vcmpgtu2(v.y & 0x7FFF7FFFu, inf2) |
          __vcmpgtu2(v.z & 0x7FFF7FFFu, inf2) | __vcmpgtu2(v.w & 0x7FFF7FFFu, inf2)) != 0;
}

__global__ void __launch_bounds__(kPtThreads) tensor_amax_kernel(const uint4* __restrict__ x,
                                                                 int64_t nvec,
                                                                 unsigned int* amax_bits) {
  uint32_t m2 = 0;
  const int64_t stride = (int64_t)gridDim.x * kPtThreads;
  int64_t i = (int64_t)blockIdx.x * kPtThreads + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {  // four 16-byte loads in flight
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ld_stream_v4(x + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) m2 = __vmaxu2(m2, mag_max8(v[u]));
  }
  for (; i < nvec; i += stride) m2 = __vmaxu2(m2, mag_max8(ld_stream_v4(x + i)));
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = __reduce_max_sync(kFull, m);
  __shared__ uint32_t red[kPtThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    uint32_t r = lane < kPtThreads / 32 ? red[lane] : 0u;
    r = __reduce_max_sync(kFull, r);
    if (lane == 0 && r != 0u) atomicMax(amax_bits, r << 16);
  }
}

__global__ void __launch_bounds__(kPtThreads) tensor_quant_kernel(const uint4* __restrict__ x,
                                                                  int64_t nvec,
                                                                  uint2* __restrict__ q,
                                                                  const float* amax_word,
                                                                  float* __restrict__ bcast,
                                                                  int64_t n_bcast) {
  const uint32_t abits = __float_as_uint(*amax_word);
  const GroupScale g = make_scale(abits, abits >= 0x7F800000u, false);
  GroupScale g_slow = g;
  g_slow.fast = false;
  const int64_t stride = (int64_t)gridDim.x * kPtThreads;
  const int64_t t0 = (int64_t)blockIdx.x * kPtThreads + threadIdx.x;
  int64_t i = t0;
  for (; i + stride < nvec; i += 2 * stride) {
    const uint4 v0 = ld_stream_v4(x + i), v1 = ld_stream_v4(x + i + stride);
    q[i] = codes_bf16x8(v0, has_nan8(v0) ? g_slow : g);
    q[i + stride] = codes_bf16x8(v1, has_nan8(v1) ? g_slow : g);
  }
  for (; i < nvec; i += stride) {
    const uint4 v = ld_stream_v4(x + i);
    q[i] = codes_bf16x8(v, has_nan8(v) ? g_slow : g);
  }
  for (int64_t j = t0; j < n_bcast; j += stride) bcast[j] = g.s;
}

__global__ void tensor_scale_finalize_kernel(float* scale_word) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *scale_word = group_scale(*scale_word);
}

// ---------------------------------------------------------------------------
// The transposing quantizers (128x1 tiles written transposed) are ops of the
// same streaming scheme.  A team (8 warps; 4 for the E4M3 re-tiling) turns
// one input tile into a 128 x 128 tile of output codes (output rows = input columns, 128 tokens
// each) and its 128 scales; it writes them into a staging buffer in its
// shared-memory scratch, and one thread stores both with bulk copies (a 2-D
// tensor store for the codes, a 512-byte copy for the scales).  The staging
// layout is the tensor map's 128-byte swizzle: 16-byte chunk c of row k sits
// at chunk c ^ (k % 8).  Each thread writes 16-byte chunks of several output
// rows; the lanes pick the order of their rows so that every group of 8
// lanes writes 8 different (k % 8) rows at once, which keeps the writes free
// of bank conflicts.
// ---------------------------------------------------------------------------

// Q1T (and, with DUAL, Q1 of the same tile): 128x1 tiles of a bf16
// activation (128 consecutive rows of one column), written transposed; with
// DUAL also the 1x128 tiles of the same rows, as Q1 writes them (grad_out
// quantized both ways from one read, page P2, paragraph 1).
// Team thread (cp, part): column pair cp (0..63) and rows 32 part ..
// 32 part + 31 of the 128 x 128 tile.
template <bool DUAL>
struct Q1TS {
  static constexpr int kStageBytes = 128 * 256;
  static constexpr int kStages = 4;
  static constexpr int kTeams = 2;
  static constexpr bool kBulkStores = true;
  static constexpr int kOffScales = 128 * 128;
  static constexpr int kOffRed = kOffScales + 128 * 4;
  static constexpr int kOffNr = kOffRed + 2 * 4 * 64 * 4;
  // DUAL: per tile row (s, s, -1/s, -1/s) of its 1x128 group (-1/s = 0 off
  // the fast path), from the lanes that made the scale to the whole half-warp
  static constexpr int kOffRowS = kOffNr + 128 * 4;
  static constexpr int kScratchBytes = kOffRowS + (DUAL ? 128 * 16 : 0);
  static constexpr uint32_t kTx = kStageBytes;
  struct Params {
    CUtensorMap map_out;  // qT [K][M] bytes, 128 x 128 box, 128-byte swizzle (64-byte aligned)
    uint8_t* q;           // DUAL: [M][K]
    float* s;             // DUAL: [K/128][M]
    float* sT;            // [M/128][K]
    int M, K, KB, num_tiles;
  };
  __device__ static void issue(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile,
                               const Params& p) {
    ptx::tma_load_2d(dst, map, bar, (tile % p.KB) * kGroup, (tile / p.KB) * kGroup);
  }
  __device__ static void consume(const uint8_t* stage, int tile, const Params& p,
                                 const Team& tm) {
    const int kb = tile % p.KB, mb = tile / p.KB;
    const int64_t k0 = (int64_t)kb * kGroup, m0 = (int64_t)mb * kGroup;
    const int t = tm.tid;
    const uint32_t* tw = reinterpret_cast<const uint32_t*>(stage);
    const int cp = t & 63, part = t >> 6;
    if constexpr (DUAL) {
      // 1x128 tiles first (their registers are free again before the 128x1
      // pass): each group of 8 lanes owns rows g8 + 32 i (i < 4), and lane
      // l8 holds elements 8 l8 .. 8 l8 + 7 and 64 + 8 l8 .. 64 + 8 l8 + 7 of
      // each (a warp's 16-byte reads then cover its four rows' halves
      // without bank conflicts).  The row maxima reduce two rows to a
      // shuffle over the group's 8 lanes; lane i (< 4) makes row i's scale
      // and leaves it, with the packed quotient operands, in a per-row
      // table that the group reads back.
      const int g8 = t >> 3, l8 = t & 7;
      uint4 v[8];
      const uint4* st = reinterpret_cast<const uint4*>(stage);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = st[(g8 + 32 * i) * 16 + l8];
        v[2 * i + 1] = st[(g8 + 32 * i) * 16 + 8 + l8];
      }
      uint32_t mj, pj;
      q1_row_max8(v, l8, mj, pj);
      float4* rs = reinterpret_cast<float4*>(tm.scratch + kOffRowS);
      bool fast = true;
      if (l8 < 4) {
        const GroupScale g = make_scale(mj, pj >= kBf16Inf, true);
        const float n = g.fast ? g.nr : 0.0f;
        const int r = g8 + 32 * l8;
        rs[r] = make_float4(g.s, g.s, n, n);
        p.s[(int64_t)kb * p.M + m0 + r] = g.s;
        fast = g.fast;
      }
      __syncwarp();
      uint8_t* qrow = p.q + (m0 + g8) * p.K + k0 + l8 * 8;
      if (__all_sync(kFull, fast)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 c = rs[g8 + 32 * i];
          const float2 s2 = make_float2(c.x, c.y), n2 = make_float2(c.z, c.w);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 x = v[2 * i + h];
            *reinterpret_cast<uint2*>(qrow + (int64_t)32 * i * p.K + 64 * h) =
                make_uint2(codes_bf16x4_fast(x.x, x.y, s2, n2), codes_bf16x4_fast(x.z, x.w, s2, n2));
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          GroupScale g;
          g.s = rs[g8 + 32 * i].x;
          g.nr = rs[g8 + 32 * i].z;
          g.fast = g.nr != 0.0f;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            *reinterpret_cast<uint2*>(qrow + (int64_t)32 * i * p.K + 64 * h) = codes_bf16x8(v[2 * i + h], g);
        }
      }
    }
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = tw[(part * 32 + i) * 64 + cp];
    release_stage(tm.empty, tm.lane);
    // 128x1 tiles: the column pair's maxima over this thread's 32 rows, the
    // NaN-free maxima recounted only where a NaN was seen
    uint32_t mp = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) mp = mag_pair_max(mp, w[i]);
    uint32_t mc = mp;
    if (pair_has_nan(mp)) {
      mc = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) mc = mag_pair_max_no_nan(mc, w[i]);
    }
    uint8_t* scr = tm.scratch;
    uint32_t* red = reinterpret_cast<uint32_t*>(scr + kOffRed);  // [2][4][64]
    red[part * 64 + cp] = mp;
    red[256 + part * 64 + cp] = mc;
    team_stage_wait(tm);
    ptx::named_barrier(tm.bar, tm.threads);
    // Each column's scale is made once: team warp tw8 finishes columns
    // 16 tw8 .. 16 tw8 + 15 (lanes 16..31 repeat lanes 0..15) and writes s
    // to the scales staging (the previous tile's bulk store has read it) and
    // -1/s (0 off the fast path) beside it.
    float* sc = reinterpret_cast<float*>(scr + kOffScales);
    float* nr = reinterpret_cast<float*>(scr + kOffNr);
    {
      const int col = 16 * (t >> 5) + (t & 15), pr = col >> 1, sh = (col & 1) * 16;
      uint32_t mpa = 0, mca = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        mpa = __vmaxu2(mpa, red[q * 64 + pr]);
        mca = __vmaxu2(mca, red[256 + q * 64 + pr]);
      }
      const GroupScale gc = make_scale((mca >> sh) & 0xFFFFu, ((mpa >> sh) & 0xFFFFu) >= kBf16Inf, true);
      if ((t & 31) < 16) {
        sc[col] = gc.s;
        nr[col] = gc.fast ? gc.nr : 0.0f;
      }
    }
    ptx::named_barrier(tm.bar, tm.threads);
    // The thread's two columns in the order it stages them: lanes with
    // (cp / 4) odd take the odd column first, which spreads each warp's
    // staging writes over all banks.
    const uint32_t hi_first = (cp >> 2) & 1;
    const uint32_t sel_a = hi_first ? 0x7632u : 0x5410u, sel_b = hi_first ? 0x5410u : 0x7632u;
    const int ka = 2 * cp + (int)hi_first, kb2 = 2 * cp + 1 - (int)hi_first;
    GroupScale ga, gb;
    ga.s = sc[ka];
    ga.nr = nr[ka];
    ga.fast = ga.nr != 0.0f;
    gb.s = sc[kb2];
    gb.nr = nr[kb2];
    gb.fast = gb.nr != 0.0f;
    uint32_t oa[8], ob[8];
    if (ga.fast && gb.fast) {
      const float2 sa2 = make_float2(ga.s, ga.s), na2 = make_float2(ga.nr, ga.nr);
      const float2 sb2 = make_float2(gb.s, gb.s), nb2 = make_float2(gb.nr, gb.nr);
#pragma unroll
      for (int i = 0; i < 32; i += 4) {  // rows i .. i + 3 of each column
        oa[i >> 2] = codes_bf16x4_fast(__byte_perm(w[i], w[i + 1], sel_a),
                                       __byte_perm(w[i + 2], w[i + 3], sel_a), sa2, na2);
        ob[i >> 2] = codes_bf16x4_fast(__byte_perm(w[i], w[i + 1], sel_b),
                                       __byte_perm(w[i + 2], w[i + 3], sel_b), sb2, nb2);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        oa[i >> 2] = codes_bf16x4(__byte_perm(w[i], w[i + 1], sel_a),
                                  __byte_perm(w[i + 2], w[i + 3], sel_a), ga);
        ob[i >> 2] = codes_bf16x4(__byte_perm(w[i], w[i + 1], sel_b),
                                  __byte_perm(w[i + 2], w[i + 3], sel_b), gb);
      }
    }
    // output rows ka and kb2, chunks 2 part and 2 part + 1
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      stage_chunk(scr, ka, 2 * part + h, make_uint4(oa[4 * h], oa[4 * h + 1], oa[4 * h + 2], oa[4 * h + 3]));
      stage_chunk(scr, kb2, 2 * part + h, make_uint4(ob[4 * h], ob[4 * h + 1], ob[4 * h + 2], ob[4 * h + 3]));
    }
    team_stage_store(tm, &p.map_out, scr, sc, (int)m0, (int)k0, p.sT + (int64_t)mb * p.K + k0);
  }
};

// Two f16 (low half first) -> two exact floats.
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h2) {
  float lo, hi;
  asm("{.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;}"
      : "=f"(lo), "=f"(hi) : "r"(h2));
  return make_float2(lo, hi);
}

// Four E5M6 codes (48 bits: lo word and the next 16 bits) of one row,
// dequantized with that row's scale: one round-to-nearest multiply each.
// An E5M6 code is an IEEE half with its mantissa cut from 10 bits to 6
// (same sign, 5-bit exponent with bias 15, subnormals, Inf and NaN), so a
// code shifted left by 4 is the half of the same value: two codes go into
// one f16x2 word by shifts and masks, and the half -> float conversion is
// exact.
__device__ __forceinline__ void dequant4_e5m6(uint32_t lo, uint32_t hi16, float s,
                                              float (&o)[4]) {
  // codes 0, 1 at bits 0..11 and 12..23 of lo; codes 2, 3 at bits 24..35
  // and 36..47 of the 48-bit value {hi16:lo}
  const uint32_t h01 = ((lo << 4) & 0x0000FFF0u) | ((lo << 8) & 0xFFF00000u);
  const uint32_t h23 = (__funnelshift_r(lo, hi16, 20) & 0x0000FFF0u) | ((hi16 << 16) & 0xFFF00000u);
  const float2 s2 = make_float2(s, s);
  const float2 a = ptx::mul2_rn(f16x2_to_f32x2(h01), s2);
  const float2 b = ptx::mul2_rn(f16x2_to_f32x2(h23), s2);
  o[0] = a.x;
  o[1] = a.y;
  o[2] = b.x;
  o[3] = b.y;
}

// Q3: 1x128 -> 128x1 re-tiling of cached codes.  A stage holds a tile of
// 128 rows (one 128-token group) x 128 columns (one K-group) of codes and
// its 128 row scales (E4M3 codes, or with E5 the packed 12-bit E5M6 cache).
// Team thread (cq, part): columns 4 cq .. 4 cq + 3, rows kRows part ..
// kRows part + kRows - 1 (two teams of 8 warps and 16 rows a thread for the
// E5M6 cache; four teams of 4 warps and 32 rows for E4M3).  The column
// maxima propagate NaN (max.NaN); only a column that holds a NaN has its
// NaN-free maximum counted again.
template <bool E5>
struct Q3S {
  static constexpr int kRowBytes = E5 ? 192 : 128;
  static constexpr int kCodeBytes = 128 * kRowBytes;
  static constexpr int kStageBytes = kCodeBytes + 128 * 4;
  static constexpr int kStages = E5 ? 4 : 8;
  static constexpr int kTeams = E5 ? 2 : 4;
  static constexpr int kTeamWarps = kConsumerWarps / kTeams;
  static constexpr int kRows = 128 / kTeamWarps;  // rows of a tile per thread
  static constexpr bool kBulkStores = true;
  static constexpr int kOffScales = 128 * 128;
  static constexpr int kOffRed = kOffScales + 128 * 4;
  static constexpr int kOffNr = kOffRed + 2 * kTeamWarps * 128 * 4;
  static constexpr int kScratchBytes = kOffNr + 128 * 4;
  static constexpr uint32_t kTx = kStageBytes;
  struct Params {
    CUtensorMap map_out;  // qT [K][M] bytes, 128 x 128 box, 128-byte swizzle (64-byte aligned)
    const float* s;       // [K/128][M]
    float* sT;            // [M/128][K]
    int M, K, KB, num_tiles;
  };
  __device__ static void issue(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile,
                               const Params& p) {
    const int kb = tile % p.KB, mb = tile / p.KB;
    ptx::tma_load_2d(dst, map, bar, kb * kRowBytes, mb * kGroup);
    ptx::bulk_load(dst + kCodeBytes, p.s + (int64_t)kb * p.M + (int64_t)mb * kGroup, 128 * 4,
                   bar);
  }
  // Codes of every column slot j for 16 rows, four rows (4h .. 4h + 3) to a
  // word, into staging row 4 cq + a[j], 16-byte chunk `chunk`.  pw holds the
  // 16 rows' codes as row-pair words (rows16 below); sp[r2] the scales of
  // rows 2 r2 and 2 r2 + 1.  kAllFast: every slot's group takes the
  // reciprocal-based quotient (the per-slot test folds away).
  template <bool kAllFast>
  __device__ __forceinline__ static void code_pass(const uint32_t (&pw)[16], const float2 (&sp)[8],
                                                   const GroupScale (&g)[4], const uint32_t (&a)[4],
                                                   uint8_t* scr, int cq, int chunk) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      GroupScale gj = g[j];
      if (kAllFast) gj.fast = true;
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t wa = pw[4 * h + (j >> 1)], wb = pw[4 * h + 2 + (j >> 1)];
        const float2 xa = ptx::mul2_rn(e4m3x2_decode((j & 1) ? wa >> 16 : wa), sp[2 * h]);
        const float2 xb = ptx::mul2_rn(e4m3x2_decode((j & 1) ? wb >> 16 : wb), sp[2 * h + 1]);
        o[h] = codes_f32x4(xa.x, xa.y, xb.x, xb.y, gj);
      }
      stage_chunk(scr, 4 * cq + a[j], chunk, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }

  // 16 rows' codes from the stage as row-pair words: pw[2 r2] holds slots
  // 0, 1 and pw[2 r2 + 1] slots 2, 3 of rows 2 r2, 2 r2 + 1 (tw and s4p
  // point at the first row's word and scales).
  __device__ __forceinline__ static void rows16(const uint32_t* tw, const float4* s4p,
                                                uint32_t sel01, uint32_t sel23, uint32_t (&pw)[16],
                                                float2 (&sp)[8]) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float4 s4 = s4p[h];
      sp[2 * h] = make_float2(s4.x, s4.y);
      sp[2 * h + 1] = make_float2(s4.z, s4.w);
    }
#pragma unroll
    for (int r2 = 0; r2 < 8; ++r2) {
      const uint32_t w0 = tw[(2 * r2) * 32], w1 = tw[(2 * r2 + 1) * 32];
      pw[2 * r2] = __byte_perm(w0, w1, sel01);
      pw[2 * r2 + 1] = __byte_perm(w0, w1, sel23);
    }
  }

  // E4M3 cache.  A byte permute gathers the codes of two consecutive rows
  // in one column into one 16-bit pair, so that every packed FP32 pair
  // (dequantization, quotient, encoding) holds rows (i, i + 1) of one
  // column: the row scales pair up straight from the stage, and the two
  // codes come out adjacent in the transposed output.  Column slot j of a
  // lane holds its column (j + rot) % 4 (rot = (cq / 2) % 4), which spreads
  // each warp's staging writes over all banks.  Teams of four warps (one
  // per SM sub-partition) take 32 rows a thread, read in blocks of 16 rows,
  // once for the column maxima and again for the codes.
  __device__ static void consume_e4m3(const uint8_t* stage, int tile, const Params& p,
                                      const Team& tm) {
    const int kb = tile % p.KB, mb = tile / p.KB;
    const int64_t k0 = (int64_t)kb * kGroup, m0 = (int64_t)mb * kGroup;
    const int cq = tm.tid & 31, part = tm.tid >> 5;
    const uint32_t rot = (cq >> 1) & 3;
    const uint32_t a[4] = {rot, (rot + 1) & 3, (rot + 2) & 3, (rot + 3) & 3};
    // __byte_perm(w_i, w_i+1, sel): bytes (w_i[a], w_i+1[a], w_i[a'], w_i+1[a'])
    const uint32_t sel01 = a[0] | ((a[0] + 4) << 4) | (a[1] << 8) | ((a[1] + 4) << 12);
    const uint32_t sel23 = a[2] | ((a[2] + 4) << 4) | (a[3] << 8) | ((a[3] + 4) << 12);
    const uint32_t* tw = reinterpret_cast<const uint32_t*>(stage) + part * kRows * 32 + cq;
    const float4* s4p = reinterpret_cast<const float4*>(stage + kCodeBytes) + part * (kRows / 4);
    float mn[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // per slot, NaN-propagating
#pragma unroll
    for (int b = 0; b < kRows / 16; ++b) {
      uint32_t pw[16];
      float2 sp[8];
      rows16(tw + b * 16 * 32, s4p + b * 4, sel01, sel23, pw, sp);
#pragma unroll
      for (int r2 = 0; r2 < 8; ++r2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = pw[2 * r2 + (j >> 1)];
          const float2 x = ptx::mul2_rn(e4m3x2_decode((j & 1) ? w >> 16 : w), sp[r2]);
          mn[j] = fmax_abs_nan(fmax_abs_nan(mn[j], x.x), x.y);
        }
      }
    }
    float mc[4] = {mn[0], mn[1], mn[2], mn[3]};
    if (mn[0] != mn[0] || mn[1] != mn[1] || mn[2] != mn[2] || mn[3] != mn[3]) {
      mc[0] = mc[1] = mc[2] = mc[3] = 0.0f;
#pragma unroll 1
      for (int b = 0; b < kRows / 16; ++b) {
        uint32_t pw[16];
        float2 sp[8];
        rows16(tw + b * 16 * 32, s4p + b * 4, sel01, sel23, pw, sp);
#pragma unroll
        for (int r2 = 0; r2 < 8; ++r2) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t w = pw[2 * r2 + (j >> 1)];
            const float2 x = ptx::mul2_rn(e4m3x2_decode((j & 1) ? w >> 16 : w), sp[r2]);
            mc[j] = fmaxf(mc[j], fmaxf(fabsf(x.x), fabsf(x.y)));
          }
        }
      }
    }
    uint8_t* scr = tm.scratch;
    float* red = reinterpret_cast<float*>(scr + kOffRed);  // [2][kTeamWarps][128]
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      red[part * 128 + 4 * cq + a[j]] = mn[j];
      red[kTeamWarps * 128 + part * 128 + 4 * cq + a[j]] = mc[j];
    }
    team_stage_wait(tm);
    ptx::named_barrier(tm.bar, tm.threads);
    float* sc = reinterpret_cast<float*>(scr + kOffScales);
    float* nr = reinterpret_cast<float*>(scr + kOffNr);
    column_scales(red, sc, nr, part, cq);
    ptx::named_barrier(tm.bar, tm.threads);
    GroupScale g[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      g[j].s = sc[4 * cq + a[j]];
      g[j].nr = nr[4 * cq + a[j]];
      g[j].fast = g[j].nr != 0.0f;
    }
    const bool all_fast = g[0].fast && g[1].fast && g[2].fast && g[3].fast;
#pragma unroll 1
    for (int b = 0; b < kRows / 16; ++b) {
      uint32_t pw[16];
      float2 sp[8];
      rows16(tw + b * 16 * 32, s4p + b * 4, sel01, sel23, pw, sp);
      if (all_fast)
        code_pass<true>(pw, sp, g, a, scr, cq, part * (kRows / 16) + b);
      else
        code_pass<false>(pw, sp, g, a, scr, cq, part * (kRows / 16) + b);
    }
    release_stage(tm.empty, tm.lane);
    team_stage_store(tm, &p.map_out, scr, sc, (int)m0, (int)k0, p.sT + (int64_t)mb * p.K + k0);
  }

  // Each column's scale is made once: warp `part` finishes columns
  // C part .. C part + C - 1 (C = 128 / kTeamWarps; with C = 16 lanes 16..31
  // repeat lanes 0..15) from the team's partial maxima red[2][kTeamWarps][128],
  // and writes s to the scales staging (which the previous tile's bulk store
  // has read, see team_stage_wait) and -1/s (0 off the fast path) beside it.
  __device__ static void column_scales(const float* red, float* sc, float* nr, int part, int cq) {
    constexpr int C = 128 / kTeamWarps;
    const int col = C * part + (cq % C);
    float a = 0.0f, b = 0.0f;  // a is NaN if the column holds a NaN
#pragma unroll
    for (int q = 0; q < kTeamWarps; ++q) {
      a = fmax_abs_nan(a, red[q * 128 + col]);
      b = fmaxf(b, red[kTeamWarps * 128 + q * 128 + col]);
    }
    const GroupScale gc = make_scale(__float_as_uint(b), !(a < __uint_as_float(kF32Inf)), false);
    if (cq < C) {
      sc[col] = gc.s;
      nr[col] = gc.fast ? gc.nr : 0.0f;
    }
  }

  __device__ static void consume(const uint8_t* stage, int tile, const Params& p,
                                 const Team& tm) {
    if constexpr (E5)
      consume_e5m6(stage, tile, p, tm);
    else
      consume_e4m3(stage, tile, p, tm);
  }

  // E5M6 cache: 12-bit codes, four per 48 bits of a row.
  __device__ static void consume_e5m6(const uint8_t* stage, int tile, const Params& p,
                                      const Team& tm) {
    const int kb = tile % p.KB, mb = tile / p.KB;
    const int64_t k0 = (int64_t)kb * kGroup, m0 = (int64_t)mb * kGroup;
    const int t = tm.tid;
    const int cq = t & 31, part = t >> 5;
    const float* srow = reinterpret_cast<const float*>(stage + kCodeBytes) + part * 16;
    // Each value is dequantized twice, for the column maxima and for the
    // codes, straight from the stage (which goes back to the producer after
    // the second pass): this keeps the kernel within the registers that 17
    // warps per SM leave (96 per thread).
    uint8_t* scr = tm.scratch;
    const uint16_t* t16 = reinterpret_cast<const uint16_t*>(stage);
    auto dq = [&](int i, float s_row, float (&xv)[4]) {
      const int h = (part * 16 + i) * 96 + 3 * cq;
      dequant4_e5m6((uint32_t)t16[h] | ((uint32_t)t16[h + 1] << 16), t16[h + 2], s_row, xv);
    };
    // column maxima that propagate NaN; the NaN-free maxima equal them
    // unless a column holds a NaN, and only then are they recounted
    float mn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      float xv[4];
      dq(i, srow[i], xv);
#pragma unroll
      for (int c = 0; c < 4; ++c) mn[c] = fmax_abs_nan(mn[c], xv[c]);
    }
    float mc[4] = {mn[0], mn[1], mn[2], mn[3]};
    if (mn[0] != mn[0] || mn[1] != mn[1] || mn[2] != mn[2] || mn[3] != mn[3]) {
      mc[0] = mc[1] = mc[2] = mc[3] = 0.0f;
#pragma unroll 1
      for (int i = 0; i < 16; ++i) {
        float xv[4];
        dq(i, srow[i], xv);
#pragma unroll
        for (int c = 0; c < 4; ++c) mc[c] = fmaxf(mc[c], fabsf(xv[c]));
      }
    }
    float* red = reinterpret_cast<float*>(scr + kOffRed);  // [2][8][128]
    static_assert(kTeamWarps == 8 && kRows == 16, "E5M6 re-tiling: teams of 8 warps");
    *reinterpret_cast<float4*>(red + part * 128 + 4 * cq) = make_float4(mn[0], mn[1], mn[2], mn[3]);
    *reinterpret_cast<float4*>(red + 1024 + part * 128 + 4 * cq) =
        make_float4(mc[0], mc[1], mc[2], mc[3]);
    team_stage_wait(tm);
    ptx::named_barrier(tm.bar, tm.threads);
    float* sc = reinterpret_cast<float*>(scr + kOffScales);
    float* nr = reinterpret_cast<float*>(scr + kOffNr);
    column_scales(red, sc, nr, part, cq);
    ptx::named_barrier(tm.bar, tm.threads);
    GroupScale g[4];
    {
      const float4 s4 = *reinterpret_cast<const float4*>(sc + 4 * cq);
      const float4 n4 = *reinterpret_cast<const float4*>(nr + 4 * cq);
      const float sv[4] = {s4.x, s4.y, s4.z, s4.w}, nv[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        g[c].s = sv[c];
        g[c].nr = nv[c];
        g[c].fast = nv[c] != 0.0f;
      }
    }
    uint32_t o[4][4];
    // all_fast: every column takes the reciprocal-based quotient (the
    // per-column test folds away)
    auto code_pass = [&](auto all_fast) {
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(srow + i);
        float x0[4], x1[4], x2[4], x3[4];
        dq(i, s4.x, x0);
        dq(i + 1, s4.y, x1);
        dq(i + 2, s4.z, x2);
        dq(i + 3, s4.w, x3);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          GroupScale gc = g[c];
          if (decltype(all_fast)::value) gc.fast = true;
          o[c][i >> 2] = codes_f32x4(x0[c], x1[c], x2[c], x3[c], gc);
        }
      }
    };
    if (g[0].fast && g[1].fast && g[2].fast && g[3].fast)
      code_pass(std::true_type());
    else
      code_pass(std::false_type());
    release_stage(tm.empty, tm.lane);
    // output rows 4 cq + c', chunk = part; lane cq writes column
    // c' = (c + cq / 2) % 4 at step c
    const int rot = (cq >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int cc = (c + rot) & 3;
      uint4 d = make_uint4(o[0][0], o[0][1], o[0][2], o[0][3]);
      if (cc == 1) d = make_uint4(o[1][0], o[1][1], o[1][2], o[1][3]);
      if (cc == 2) d = make_uint4(o[2][0], o[2][1], o[2][2], o[2][3]);
      if (cc == 3) d = make_uint4(o[3][0], o[3][1], o[3][2], o[3][3]);
      stage_chunk(scr, 4 * cq + cc, part, d);
    }
    team_stage_store(tm, &p.map_out, scr, sc, (int)m0, (int)k0, p.sT + (int64_t)mb * p.K + k0);
  }
};

int num_sms_current_device() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <class Op>
cudaError_t launch_stream(const CUtensorMap& map, const typename Op::Params& p,
                          cudaStream_t stream) {
  using L = StreamSmem<Op>;
  auto kern = stream_kernel<Op>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  int grid = num_sms_current_device();
  if (grid > p.num_tiles) grid = p.num_tiles;
  kern<<<grid, kThreads, L::kAlloc, stream>>>(map, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                   cudaStream_t stream) {
  CUtensorMap map;
  if (!make_tmap_2d(&map, x, 2, M, K, kGroup, Q1::kRows, false)) return cudaErrorInvalidValue;
  Q1::Params p;
  p.q = q;
  p.s = s;
  p.M = (int)M;
  p.K = (int)K;
  p.KB = (int)(K / kGroup);
  p.num_tiles = (int)((M + Q1::kRows - 1) / Q1::kRows) * p.KB;
  p.unused = nullptr;
  return launch_stream<Q1>(map, p, stream);
}

namespace {

// Output tensor map of a transposing quantizer: qT [K][M] bytes, 128 x 128
// boxes with the 128-byte swizzle of the staging buffers.
bool make_out_map(CUtensorMap* map, uint8_t* qT, int64_t K, int64_t M) {
  return make_tmap_2d(map, qT, 1, K, M, kGroup, kGroup, true);
}

template <bool DUAL>
cudaError_t launch_q1t(const void* x, int64_t M, int64_t K, uint8_t* qT, float* sT, uint8_t* q,
                       float* s, cudaStream_t stream) {
  CUtensorMap map;
  typename Q1TS<DUAL>::Params p;
  if (!make_tmap_2d(&map, x, 2, M, K, kGroup, kGroup, false) || !make_out_map(&p.map_out, qT, K, M))
    return cudaErrorInvalidValue;
  p.q = q;
  p.s = s;
  p.sT = sT;
  p.M = (int)M;
  p.K = (int)K;
  p.KB = (int)(K / kGroup);
  p.num_tiles = (int)(M / kGroup) * p.KB;
  return launch_stream<Q1TS<DUAL>>(map, p, stream);
}

template <bool E5>
cudaError_t launch_q3(const uint8_t* q, const float* s, int64_t M, int64_t K, uint8_t* qT,
                      float* sT, cudaStream_t stream) {
  CUtensorMap map;
  typename Q3S<E5>::Params p;
  const int64_t row_bytes = E5 ? K / 2 * 3 : K;
  if (!make_tmap_2d(&map, q, 1, M, row_bytes, Q3S<E5>::kRowBytes, kGroup, false) ||
      !make_out_map(&p.map_out, qT, K, M))
    return cudaErrorInvalidValue;
  p.s = s;
  p.sT = sT;
  p.M = (int)M;
  p.K = (int)K;
  p.KB = (int)(K / kGroup);
  p.num_tiles = (int)(M / kGroup) * p.KB;
  return launch_stream<Q3S<E5>>(map, p, stream);
}

}  // namespace

cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, uint8_t* qT, float* sT,
                                   cudaStream_t stream) {
  return launch_q1t<false>(x, M, K, qT, sT, nullptr, nullptr, stream);
}

cudaError_t launch_quant_act_dual(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                  uint8_t* qT, float* sT, cudaStream_t stream) {
  return launch_q1t<true>(x, M, K, qT, sT, q, s, stream);
}

cudaError_t launch_quant_act_and_weight(const void* x, int64_t M, int64_t K, uint8_t* q,
                                        float* s, const void* w, int64_t N, int64_t Kw,
                                        uint8_t* qw, float* sw, cudaStream_t stream) {
  Q12::Params p;
  CUtensorMap map_a;
  if (!make_tmap_2d(&map_a, x, 2, M, K, kGroup, Q1::kRows, false)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&p.map_w, w, 2, N, Kw, kGroup, kGroup, false)) return cudaErrorInvalidValue;
  p.a.q = q;
  p.a.s = s;
  p.a.M = (int)M;
  p.a.K = (int)K;
  p.a.KB = (int)(K / kGroup);
  p.a.num_tiles = (int)((M + Q1::kRows - 1) / Q1::kRows) * p.a.KB;
  p.a.unused = nullptr;
  p.w.q = qw;
  p.w.s = sw;
  p.w.qT = nullptr;
  p.w.sT = nullptr;
  p.w.N = (int)N;
  p.w.K = (int)Kw;
  p.w.KB = (int)(Kw / kGroup);
  p.w.NB = (int)(N / kGroup);
  p.w.num_tiles = p.w.NB * p.w.KB;
  p.t1 = p.a.num_tiles;
  p.num_tiles = p.a.num_tiles + p.w.num_tiles;
  return launch_stream<Q12>(map_a, p, stream);
}

cudaError_t launch_quant_weight_128x128(const void* w, int64_t N, int64_t K, uint8_t* q, float* s,
                                        uint8_t* qT, float* sT, cudaStream_t stream) {
  CUtensorMap map;
  if (!make_tmap_2d(&map, w, 2, N, K, kGroup, kGroup, false)) return cudaErrorInvalidValue;
  Q2::Params p;
  if (qT && !make_out_map(&p.map_t, qT, K, N)) return cudaErrorInvalidValue;
  p.q = q;
  p.s = s;
  p.qT = qT;
  p.sT = sT;
  p.N = (int)N;
  p.K = (int)K;
  p.KB = (int)(K / kGroup);
  p.NB = (int)(N / kGroup);
  p.num_tiles = p.NB * p.KB;
  return launch_stream<Q2>(map, p, stream);
}

cudaError_t launch_requant_1x128_to_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                          uint8_t* qT, float* sT, cudaStream_t stream) {
  return launch_q3<false>(q, s, M, K, qT, sT, stream);
}

cudaError_t launch_quant_per_tensor(const void* x, int64_t n, uint8_t* q, float* scale,
                                    float* bcast, int64_t n_bcast, cudaStream_t stream) {
  const int64_t nvec = n / 8;
  cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t max_grid = (int64_t)num_sms_current_device() * kPtCtasPerSm;
  int64_t g1 = (nvec + kPtThreads - 1) / kPtThreads;
  g1 = g1 < 1 ? 1 : (g1 > max_grid ? max_grid : g1);
  const auto* xv = static_cast<const uint4*>(x);
  tensor_amax_kernel<<<(unsigned)g1, kPtThreads, 0, stream>>>(
      xv, nvec, reinterpret_cast<unsigned int*>(scale));
  int64_t g2 = ((nvec > n_bcast ? nvec : n_bcast) + kPtThreads - 1) / kPtThreads;
  g2 = g2 < 1 ? 1 : (g2 > max_grid ? max_grid : g2);
  tensor_quant_kernel<<<(unsigned)g2, kPtThreads, 0, stream>>>(
      xv, nvec, reinterpret_cast<uint2*>(q), scale, bcast, n_bcast);
  tensor_scale_finalize_kernel<<<1, 32, 0, stream>>>(scale);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_e5m6(const void* x, int64_t M, int64_t K, uint8_t* e5, float* s5,
                                  uint8_t* q, float* s, cudaStream_t stream) {
  CUtensorMap map;
  if (!make_tmap_2d(&map, x, 2, M, K, kGroup, Q1E5::kRows, false)) return cudaErrorInvalidValue;
  Q1E5::Params p;
  p.e5 = e5;
  p.s5 = s5;
  p.q = q;
  p.s = s;
  p.M = (int)M;
  p.K = (int)K;
  p.KB = (int)(K / kGroup);
  p.num_tiles = (int)((M + Q1E5::kRows - 1) / Q1E5::kRows) * p.KB;
  return launch_stream<Q1E5>(map, p, stream);
}

cudaError_t launch_requant_e5m6_to_128x1(const uint8_t* e5, const float* s5, int64_t M, int64_t K,
                                         uint8_t* qT, float* sT, cudaStream_t stream) {
  return launch_q3<true>(e5, s5, M, K, qT, sT, stream);
}

// The quantizers' error word, taken like the GEMM's (enqueue_take_gemm_error).
__global__ void take_quant_error_kernel(unsigned int* dst) {
  *dst = atomicExch(&g_quant_error, 0u);
}

cudaError_t enqueue_take_quant_error(unsigned int* dst, cudaStream_t stream) {
  take_quant_error_kernel<<<1, 1, 0, stream>>>(dst);
  return cudaGetLastError();
}

}  // namespace fp8bs
