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
//   * persistent CTAs, one per SM, each computing 128 x BN output tiles
//     (BN = 128 ... 256, chosen per shape to limit wave quantization), or,
//     as a CTA pair (tcgen05 cta_group::2, a cluster of two), 256 x BN tiles
//     whose MMAs span both SMs: each CTA loads its own 128 rows of A and its
//     own half of the B tile, and the tensor cores read the peer's half
//     directly, which halves the shared-memory traffic of B per MAC;
//   * no TMA load is multicast: every copy lands only in the shared memory
//     of the CTA that issues it;
//   * warp 0 -- TMA producer: A and B K-group tiles (128 B rows, 128-byte
//     swizzle) into a STAGES-deep shared-memory ring (mbarrier full/empty;
//     for a pair, both CTAs' copies complete on the leader's full barrier
//     and the leader's MMA commit frees the stage in both CTAs);
//   * warp 1 -- MMA issuer: per K-group, four tcgen05.mma kind::f8f6f4
//     (K = 32 each) into one of the TMEM partial buffers, then
//     tcgen05.commit to free the smem stage and to publish the partial;
//   * warp 2 -- scale loader: the K-group's 128 row scales of A and the
//     tile's B scales into a small shared ring, by cp.async completing on an
//     mbarrier, so it never waits for memory itself;
//   * warps 4..11 -- promotion: each owns 32 TMEM lanes (rows) and half the
//     tile's columns, keeps the FP32 accumulator in registers (setmaxnreg
//     moves registers from warps 0-3 to these when BN > 128), and per
//     K-group does acc += P_g * (sa * sb) while the tensor core already
//     computes the next group's partial into the other TMEM buffer (the
//     "overlapping of the two operations" of P3 paragraph 4 / P4 paragraph 1);
//     the epilogue converts to BF16 (RNE) or keeps FP32 and stores.
//   * the per-K-group hand-off is the cost centre: the MMA issuer sleeps
//     in its barrier waits (a polling thread takes issue slots and shared
//     memory bandwidth from the promotion warps beside it), and TMEM buffers
//     are released with relaxed arrivals (the data is already in registers);
//   * launched as a programmatic dependent: barriers, TMEM and tensor maps
//     are set up while the previous kernel on the stream finishes;
//   * every mbarrier wait is bounded (globaltimer); on expiry the kernel
//     sets a device error word and an abort flag, every role winds down,
//     in-flight copies and MMAs are drained (bounded) and TMEM is freed.
//
// The un-promoted variant (PROMOTE = false) keeps the whole K inside one
// TMEM accumulator and applies K-group 0's scales once at the end: the
// measurement of what tensor-core-only accumulation costs (P1 paragraph 4).
#include <atomic>
#include <cmath>
#include <mutex>

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
constexpr int kFirstPromoWarp = 4;  // warps 0..3 control, 4.. promotion
// Scales reach the promotion warps through a ring of kScaleSlots slots of
// kScaleGroup K-groups each: one barrier wait and one release per slot, not
// per K-group.
constexpr int kScaleGroup = 4;
constexpr int kScaleSlots = 2;
constexpr int kScaleEntries = kScaleGroup * kScaleSlots;
constexpr int kSmemLimit = 232448;  // 227 KB: the opt-in maximum per block
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
  float* c_scales;  // E4M3 output: [N/128][M]
  int M, N, K, KB;
  int num_m_units, num_units;  // a unit = one 128 x BN tile, or a pair's 256 x BN tile
  int num_n_units, group_m;     // unit columns; unit rows per group (tile order)
  int skip_iter;
  // Stream-K: units below sk_begin go whole to CTA groups g, g + G, ...
  // (G = num_groups); the S = sk_iters K-groups of units sk_begin..
  // (unit-major) are split evenly: with S = q G + r (sk_q, sk_r), group g
  // takes q + 1 of them if g < r, else q, in group order.  A unit split over
  // several groups is summed through ws (each group's FP32 share) and ws_cnt
  // (one arrival counter per unit, CTA and promotion warp); sk_begin ==
  // num_units turns it off.
  int sk_begin, num_groups;
  int sk_iters, sk_q, sk_r;
  float* ws;
  unsigned int* ws_cnt;
};

// Unit u's row of units and column of tiles.  Units are taken in groups of
// group_m unit rows, the row changing fastest within a group: the units in
// flight at one time then share a few A row panels and B column panels in
// L2.  With the row changing fastest over all of M, every wave would stream
// the whole of A from HBM once (measured at the 8192 x 8192 x 16384 stress
// shape: 2.12 GB read per launch against 0.28 GB of operands).
__device__ __forceinline__ void unit_coords(const Params& p, int u, int& mu, int& nt) {
  const int per_group = p.group_m * p.num_n_units;
  const int grp = u / per_group, r = u - grp * per_group;
  const int first = grp * p.group_m;
  const int gm = min(p.num_m_units - first, p.group_m);
  mu = first + r % gm;
  nt = r / gm;
}

// First stream-K iteration of CTA group g's share.
__device__ __forceinline__ int sk_share_begin(const Params& p, int g) {
  return g * p.sk_q + min(g, p.sk_r);
}

// The CTA group whose share holds stream-K iteration `it`.
__device__ __forceinline__ int sk_owner(const Params& p, int it) {
  const int big = p.sk_r * (p.sk_q + 1);  // iterations of the r larger shares
  return it < big ? it / (p.sk_q + 1) : p.sk_r + (it - big) / p.sk_q;
}

// The work of CTA group g, one item at a time: whole units g, g + G, ...
// below sk_begin, then its stream-K share as segments (unit u, K-groups
// kb0 .. kb1 - 1).  Every role of the CTA walks the same items.
struct WorkIter {
  int u, kb0, kb1;
  int it, it_end;
  bool valid;
  __device__ __forceinline__ WorkIter(const Params& p, int g) {
    u = g;
    kb0 = 0;
    kb1 = p.KB;
    it = sk_share_begin(p, g);
    it_end = sk_share_begin(p, g + 1);
    valid = true;
    if (u >= p.sk_begin) start_sk(p);
  }
  __device__ __forceinline__ void start_sk(const Params& p) {
    valid = it < it_end;
    if (!valid) return;
    u = p.sk_begin + it / p.KB;
    kb0 = it % p.KB;
    kb1 = min(p.KB, kb0 + (it_end - it));
  }
  __device__ __forceinline__ void next(const Params& p) {
    if (u < p.sk_begin) {
      u += p.num_groups;
      kb0 = 0;
      kb1 = p.KB;
      if (u >= p.sk_begin) start_sk(p);
      return;
    }
    it += kb1 - kb0;
    start_sk(p);
  }
  // true when this is the group's last item
  __device__ __forceinline__ bool last(const Params& p) const {
    WorkIter n = *this;
    n.next(p);
    return !n.valid;
  }
};

// Workspace slot of group g's segment of unit u: 2 g for the first segment
// of g's stream-K share, 2 g + 1 for its last (a share holds at most these
// two partial segments; whole units between them need no slot).
__device__ __forceinline__ int sk_slot(const Params& p, int g, int u) {
  return u == p.sk_begin + sk_share_begin(p, g) / p.KB ? 2 * g : 2 * g + 1;
}

// Bounded wait.  Returns false when this wait expired (the error word and
// the CTA's abort flag get set) or another role already aborted.
// With SUSPEND the waiting thread sleeps in the barrier (at most 20 us per
// try, so the time limit below still holds) instead of polling.
template <bool SUSPEND = false>
__device__ __forceinline__ bool try_wait(uint32_t addr, uint32_t parity) {
  if constexpr (SUSPEND)
    return ptx::mbar_try_wait_suspend<20000>(addr, parity);
  else
    return ptx::mbar_try_wait(addr, parity);
}

template <bool SUSPEND = false>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int site) {
  const uint32_t addr = ptx::smem_addr(bar);
  // a phase that has already completed is seen by one non-blocking test
  if (ptx::mbar_test_wait(addr, parity)) return true;
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (try_wait<SUSPEND>(addr, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (try_wait<SUSPEND>(addr, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      atomicOr(&g_device_error, site);
      return false;
    }
  }
}

// PW promotion warps (8, 12 or 16) share the tile's columns: each owns 32
// TMEM lanes (rows) and kCols = BN / (PW / 4) columns.  Per K-group each
// promotion thread spends one FP32 operation per element with block B
// scales and two with per-column B scales (fl(p sb) then fma with sa).
// With per-column scales the promotion warps bound the kernel (with the
// MMAs taken out the 256 x 256 pair runs at the same speed; the MMA issuer
// waits for the TMEM buffer most of each K-group); with block scales the
// chain is balanced: the MMA issuer waits in turn for operands, for the
// buffer and for the tensor pipe.
template <int BN, bool PAIR, int PW>
struct Cfg {
  static constexpr int CM = PAIR ? 2 : 1;  // CTAs per cluster
  static_assert(PW == 8 || PW == 12 || PW == 16, "promotion warps");
  static constexpr int kPromoWarps = PW;
  static constexpr int kThreads = 32 * (kFirstPromoWarp + PW);
  static constexpr int kCols = BN / (PW / 4);
  static_assert(kCols % 16 == 0, "columns per promotion warp");
  // 16 warps: each reads its steps into one register buffer (the four warps
  // of a sub-partition overlap one another's reads).  Otherwise a warp with
  // at most 64 columns reads its whole partial at once and hands the buffer
  // back before its FMAs, and wider warps read in double-buffered steps.
  static constexpr bool kSingleBuf = PW == 16;
  static constexpr bool kLoadAll = !kSingleBuf && kCols <= 64;
  // Register split when the accumulators need more than an even share:
  // warpgroup 0 (producer, MMA, scales) keeps kCtlRegs, the promotion
  // warpgroups get kPromoRegs.  Their sum must fit in what the launch holds:
  // kThreads threads at kLaunchRegs each (65536 / kThreads, rounded down to
  // the allocation unit of 8).
  static constexpr bool kRegSplit = PW >= 12 || BN > 128;
  static constexpr int kCtlRegs = PW == 16 ? 32 : PW == 12 ? 56 : 48;
  static constexpr int kPromoRegs = PW == 16 ? 112 : PW == 12 ? 152 : 224;
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8;
  static constexpr int kSplitRegsNeeded = 128 * kCtlRegs + 32 * PW * kPromoRegs;
  static_assert(!kRegSplit || kSplitRegsNeeded <= kLaunchRegs * kThreads, "register split");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
  // B rows this CTA loads: the whole B tile, or, for a CTA pair, its own
  // half of the pair's B tile
  static constexpr int kBH = BN / CM;
  static_assert(kBH % 8 == 0, "B half must be whole 8-row swizzle atoms");
  // columns between TMEM partial buffers, and how many fit in 512 columns
  static constexpr int kTmemStride = BN <= 128 ? 128 : BN <= 160 ? 160 : 256;
  static constexpr int kTBuf = 512 / kTmemStride > 4 ? 4 : 512 / kTmemStride;
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = kBH * kBK;
  static constexpr int kScaleB = BN + 4;  // B scales per slot (tile: BN, block: <= 3)
  static constexpr int kScaleFloats = kBM + kScaleB;
  // Epilogue staging for tensor-store output: 4 KB per promotion warp (its
  // 32 rows x up to 128 bytes).
  static constexpr bool kEpiTma = kCols % 16 == 0;
  static constexpr int kEpiBytes = kEpiTma ? PW * 4096 : 0;
  static constexpr int kNumBarsMax = 2 * 8 + 2 * 4 + 2 * kScaleSlots + 1;
  static constexpr int kFixed =
      kEpiBytes + kScaleEntries * kScaleFloats * 4 + kNumBarsMax * 8 + 16 + 1024;
  static constexpr int kStagesFit = (kSmemLimit - kFixed) / (kABytes + kBBytes);
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static_assert(kStages >= 2, "shared memory");
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffEpi = kOffB + kStages * kBBytes;  // 1024-aligned (128-byte swizzle)
  static_assert(kOffEpi % 1024 == 0, "staging alignment");
  static constexpr int kOffScale = kOffEpi + kEpiBytes;
  static constexpr int kOffBar = kOffScale + kScaleEntries * kScaleFloats * 4;
  static constexpr int kNumBars = 2 * kStages + 2 * kTBuf + 2 * kScaleSlots + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
  static_assert(kAlloc <= kSmemLimit, "shared memory");
};

// The four K = 32 MMAs of one K-group (accumulating onto D unless this is
// the first K-group and `accumulate_first` is false).
template <bool PAIR>
__device__ __forceinline__ void issue_kgroup(uint32_t d, uint32_t a0, uint32_t b0, uint32_t idesc,
                                             bool accumulate_first) {
  // Each K = 32 step starts 32 bytes further into the 128-byte rows: +2 in
  // the descriptor's address field (address >> 4; no carry, since shared
  // memory addresses stay far below 2^18).
  const uint64_t ad0 = ptx::smem_desc_k128_sw128(a0);
  const uint64_t bd0 = ptx::smem_desc_k128_sw128(b0);
#pragma unroll
  for (int k = 0; k < kBK / 32; ++k) {
    const uint64_t ad = ad0 + 2u * k;
    const uint64_t bd = bd0 + 2u * k;
    const uint32_t acc = (accumulate_first || k > 0) ? 1u : 0u;
    if (PAIR)
      ptx::mma_f8f6f4_pair(d, ad, bd, idesc, acc);
    else
      ptx::mma_f8f6f4(d, ad, bd, idesc, acc);
  }
}

// Free a shared-memory stage once the MMAs reading it completed: in this
// CTA, or in both CTAs of a pair (the commit arrives on the barrier at the
// same offset in each CTA).
template <bool PAIR>
__device__ __forceinline__ void commit_stage(uint64_t* empty) {
  if (PAIR)
    ptx::tc_commit_pair_mcast(empty, 0x3);
  else
    ptx::tc_commit(empty);
}

// Hand a TMEM partial buffer back to the MMA issuer (the pair's leader).
// The caller has waited for its TMEM reads (tcgen05.wait::ld) and fenced
// them (tcgen05.fence::before_thread_sync): the data is in registers and no
// memory access needs ordering, so the arrival is relaxed.
template <bool PAIR>
__device__ __forceinline__ void release_tmem(uint64_t* tempty) {
  if (PAIR)
    ptx::mbar_arrive_cluster_relaxed(ptx::mapa(tempty, 0));
  else
    ptx::mbar_arrive_relaxed(tempty);
}

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// TMEM read steps of a promotion warp that owns kCols columns: step st
// covers columns [32 st, 32 st + width) of the warp's range, width = 32
// except a final 16.  Every load starts on a multiple of 16 columns.
template <int kCols>
struct PromoSteps {
  static_assert(kCols % 16 == 0, "columns");
  static constexpr int kSteps = (kCols + 31) / 32;
  static constexpr int width(int st) { return kCols - 32 * st < 32 ? kCols - 32 * st : 32; }
};

// acc[a0 .. a0 + kC) += P * scale for one step of kC columns that starts at
// column a0 of the warp's kCols (tile column col0 + a0).  Block scales
// change only at 128-column boundaries, which fall on multiples of 16
// columns of the warp's range; tile scales change per column.
template <int kC, int a0, bool B_TILE, int kBatch = 32>
__device__ __forceinline__ void promote_step(float* acc, const uint32_t* v, float sa_r,
                                             const float* scb, int col0, float f_lo, float f_hi,
                                             int a_split) {
  if constexpr (B_TILE) {
    // one broadcast 16-byte shared-memory read serves four columns; the
    // reads of a batch of kBatch columns are all issued before its FMAs, so
    // their latencies overlap
    const float2 sa2 = make_float2(sa_r, sa_r);
    constexpr int kB = kBatch < kC ? kBatch : kC;
    float4 sbv[kB / 4];
#pragma unroll
    for (int j = 0; j < kC; j += 4) {
      if (j % kB == 0) {
#pragma unroll
        for (int i = 0; i < kB; i += 4)
          sbv[i / 4] = *reinterpret_cast<const float4*>(scb + col0 + a0 + j + i);
      }
      const float4 sb4 = sbv[(j % kB) / 4];
      const float2 p0 = make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
      const float2 p1 = make_float2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      const float2 r0 = ptx::fma2_rn(ptx::mul2_rn(p0, make_float2(sb4.x, sb4.y)), sa2,
                                     make_float2(acc[a0 + j], acc[a0 + j + 1]));
      const float2 r1 = ptx::fma2_rn(ptx::mul2_rn(p1, make_float2(sb4.z, sb4.w)), sa2,
                                     make_float2(acc[a0 + j + 2], acc[a0 + j + 3]));
      acc[a0 + j] = r0.x;
      acc[a0 + j + 1] = r0.y;
      acc[a0 + j + 2] = r1.x;
      acc[a0 + j + 3] = r1.y;
    }
  } else {
    // the warp's columns lie in at most two 128-column blocks: factor f_lo
    // before column a_split of the warp's range, f_hi from there on (block
    // boundaries fall on multiples of 16 columns)
#pragma unroll
    for (int j0 = 0; j0 < kC; j0 += 16) {
      const float f = (a0 + j0 < a_split) ? f_lo : f_hi;
      const float2 f2 = make_float2(f, f);
#pragma unroll
      for (int j = j0; j < j0 + 16 && j < kC; j += 2) {
        const float2 pv = make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
        const float2 r = ptx::fma2_rn(pv, f2, make_float2(acc[a0 + j], acc[a0 + j + 1]));
        acc[a0 + j] = r.x;
        acc[a0 + j + 1] = r.y;
      }
    }
  }
}

// A promotion warp's FP32 share of a stream-K unit in the workspace: lane
// l's columns j .. j+3 at float4 l + 32 (j / 4) of the warp's chunk, so each
// store or load of the warp covers 512 contiguous bytes.  One base address
// and immediate offsets, and the loads one at a time (ordered volatile asm,
// each sum pinned before the next load): the share needs no registers
// beside the accumulator.
template <int kCols, int J = 0>
__device__ __forceinline__ void share_store(const float4* base, const float* acc) {
  if constexpr (J < kCols) {
    asm volatile("st.global.cg.v4.f32 [%0+%1], {%2, %3, %4, %5};" ::"l"(base), "n"(J / 4 * 512),
                 "f"(acc[J]), "f"(acc[J + 1]), "f"(acc[J + 2]), "f"(acc[J + 3])
                 : "memory");
    share_store<kCols, J + 4>(base, acc);
  }
}

// acc[J .. J+31] = the sum over groups g_first .. g_last, in that order, of
// their shares' float4s J / 4 .. J / 4 + 7 (sh(g) gives a group's base
// address): eight loads in flight per group, the batch's sums pinned before
// the next batch's loads so that at most 64 registers join the accumulator.
template <int kCols, int J = 0, class Sh>
__device__ __forceinline__ void share_sum(float* acc, const Sh& sh, int g_first, int g_last) {
  if constexpr (J < kCols) {
    constexpr int kB = (kCols - J) / 4 < 8 ? (kCols - J) / 4 : 8;  // float4s in this batch
    float4 t[kB];
#pragma unroll
    for (int i = 0; i < kB; ++i) t[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
    for (int g = g_first; g <= g_last; ++g) {
      const float4* base = sh(g);
      float4 v[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) v[i] = __ldcg(base + (J / 4 + i) * 32);
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        t[i].x += v[i].x;
        t[i].y += v[i].y;
        t[i].z += v[i].z;
        t[i].w += v[i].w;
      }
    }
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      acc[J + 4 * i] = t[i].x;
      acc[J + 4 * i + 1] = t[i].y;
      acc[J + 4 * i + 2] = t[i].z;
      acc[J + 4 * i + 3] = t[i].w;
      asm volatile("" : "+f"(acc[J + 4 * i]), "+f"(acc[J + 4 * i + 1]), "+f"(acc[J + 4 * i + 2]),
                   "+f"(acc[J + 4 * i + 3]));
    }
    share_sum<kCols, J + 4 * kB>(acc, sh, g_first, g_last);
  }
}

// Load kC columns (32 or 16) from TMEM.
template <int kC>
__device__ __forceinline__ void tmem_ld_step(uint32_t taddr, uint32_t* r) {
  static_assert(kC == 32 || kC == 16, "columns");
  if constexpr (kC == 32)
    ptx::tmem_ld_32x32b_x32(taddr, r);
  else
    ptx::tmem_ld_32x32b_x16(taddr, r);
}

// Output kinds: FP32, BF16 (round to nearest even), or E4M3 codes with one
// FP32 scale per 1x128 tile of each output row (the next layer's activation
// quantized in the epilogue).
enum : int { kOutF32 = 0, kOutBf16 = 1, kOutE4m3 = 2 };

template <int BN, bool PAIR, int PW, bool PROMOTE, int OUT, bool B_TILE>
__global__ void __launch_bounds__(32 * (kFirstPromoWarp + PW), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_c, const Params p) {
  using L = Cfg<BN, PAIR, PW>;
  constexpr int CM = L::CM;
  constexpr int kPromoWarps = L::kPromoWarps;
  constexpr int STAGES = L::kStages;
  constexpr int TBUF = L::kTBuf;
  // The MMA issuer sleeps in its barrier waits instead of polling on the
  // CTA-pair shapes and on the one-CTA shapes narrower than 256 with 8
  // promotion warps: its polling competed with the promotion warps of its
  // sub-partition, and sleeping measured +5% (128 x 224) to +16% (128 x 128)
  // and +10-15% on the pairs.  The one-CTA 256-wide and 12-warp shapes
  // measured the same either way and poll.
  constexpr bool kMmaSuspend = PAIR || (PW == 8 && BN < 256);
  constexpr int kCols = L::kCols;  // columns per promotion warp
  constexpr uint32_t kTmemCols = 512;
  // a CTA pair runs M = 256 MMAs, each CTA holding 128 rows of A and of D
  constexpr uint32_t kIdesc = ptx::idesc_e4m3_f32(PAIR ? 2 * kBM : kBM, BN);
  // bytes one stage's full barrier waits for: what lands in this CTA, or,
  // for a pair (whose leader's barrier counts both CTAs' copies), twice that
  constexpr uint32_t kStageTx = (PAIR ? 2 : 1) * (L::kABytes + L::kBBytes);

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
  const int rank = CM > 1 ? (int)ptx::cluster_ctarank() : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);
      // one MMA commit (a pair's leader commits to both CTAs)
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < TBUF; ++i) {
      ptx::mbar_init(&tfull[i], 1);
      // a pair's leader waits for both CTAs' promotion warps
      ptx::mbar_init(&tempty[i], PAIR ? 2 * kPromoWarps : kPromoWarps);
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
    if (PAIR) {  // collective: both CTAs of the pair get the same columns
      ptx::tmem_alloc_pair(tmem_base_slot, kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_base_slot, kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // a pair's barriers must be initialised before the peer's copies and
  // commits reach them
  if (PAIR) ptx::cluster_sync();
  const uint32_t tmem_base = *tmem_base_slot;
  // Launched as a programmatic dependent: everything above overlapped the
  // previous kernel's tail; its results are visible from here on.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int KB = p.KB;
  const int unit_first = blockIdx.x / CM;  // this CTA's group

  if (warp < kFirstPromoWarp) {
  // Warpgroup 0: producer, MMA issuer, scale loader (warp 3 idles).  Each
  // warpgroup changes its register allocation at the top of its own branch,
  // so that the code it runs is compiled against the new limit.
  if constexpr (L::kRegSplit) ptx::regs_dec<L::kCtlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_a);
      ptx::prefetch_tmap(&tmap_b);
      uint32_t it = 0;
      uint32_t issued_mask = 0;  // stages with a copy issued at least once
      bool ok = true;
      for (WorkIter wk(p, unit_first); ok && wk.valid; wk.next(p)) {
        int mu, nt;
        unit_coords(p, wk.u, mu, nt);
        const int mt = mu * CM + rank;
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it) {
          const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1;
          if (!wait_bar(&empty[stage], phase ^ 1, abort_flag, kErrProducer)) { ok = false; break; }
          if ((int)it == p.skip_iter) continue;  // test hook: never arrives
          if (PAIR) {
            // both CTAs' copies complete on the leader's barrier
            if (rank == 0) ptx::mbar_arrive_expect_tx(&full[stage], kStageTx);
            const uint32_t fb = ptx::mapa(&full[stage], 0);
            ptx::tma_load_2d_pair(sA + stage * L::kABytes, &tmap_a, fb, kb * kBK, mt * kBM);
            ptx::tma_load_2d_pair(sB + stage * L::kBBytes, &tmap_b, fb, kb * kBK,
                                  nt * BN + rank * L::kBH);
            issued_mask |= 1u << stage;
            continue;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], kStageTx);
          ptx::tma_load_2d(sA + stage * L::kABytes, &tmap_a, &full[stage], kb * kBK, mt * kBM);
          ptx::tma_load_2d(sB + stage * L::kBBytes, &tmap_b, &full[stage], kb * kBK, nt * BN);
          issued_mask |= 1u << stage;
        }
      }
      // Drain: wait (bounded) until the last copy issued into each stage has
      // landed, so no copy is in flight when the CTA exits.  A pair's
      // follower has no full barriers of its own: its copies complete on the
      // leader's, which the leader drains.
      const uint32_t last = (PAIR && rank != 0) ? 0 : it;
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
    // (for a CTA pair, the leader issues the pair's MMAs)
    if (lane == 0 && (!PAIR || rank == 0)) {
      uint32_t it = 0, kt = 0;
      bool ok = true;
      for (WorkIter wk(p, unit_first); ok && wk.valid; wk.next(p)) {
        if (PROMOTE) {
          for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it, ++kt) {
            // The operands usually land long before the TMEM buffer comes
            // back: wait for them first, so that once the promotion warps
            // release the buffer only the MMAs remain to be issued.
            const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1;
            if (!wait_bar<kMmaSuspend>(&full[stage], phase, abort_flag, kErrMma)) {
              ok = false;
              break;
            }
            const uint32_t a0 = ptx::smem_addr(sA + stage * L::kABytes);
            const uint32_t b0 = ptx::smem_addr(sB + stage * L::kBBytes);
            const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
            const uint32_t d = tmem_base + buf * L::kTmemStride;
            if (!wait_bar<kMmaSuspend>(&tempty[buf], tph ^ 1, abort_flag, kErrMma)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            issue_kgroup<PAIR>(d, a0, b0, kIdesc, false);
            commit_stage<PAIR>(&empty[stage]);
            if (PAIR)
              ptx::tc_commit_pair_mcast(&tfull[buf], 0x3);
            else
              ptx::tc_commit(&tfull[buf]);
          }
        } else {
          const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
          if (!wait_bar(&tempty[buf], tph ^ 1, abort_flag, kErrMma)) break;
          ptx::tc_fence_after();
          const uint32_t d = tmem_base + buf * L::kTmemStride;
          for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it) {
            const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1;
            if (!wait_bar(&full[stage], phase, abort_flag, kErrMma)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t a0 = ptx::smem_addr(sA + stage * L::kABytes);
            const uint32_t b0 = ptx::smem_addr(sB + stage * L::kBBytes);
            issue_kgroup<PAIR>(d, a0, b0, kIdesc, kb > wk.kb0);
            commit_stage<PAIR>(&empty[stage]);
          }
          if (!ok) break;
          if (PAIR)
            ptx::tc_commit_pair_mcast(&tfull[buf], 0x3);
          else
            ptx::tc_commit(&tfull[buf]);
          ++kt;
        }
      }
      // Drain: every MMA this thread issued has completed before TMEM is freed.
      if (PAIR)
        ptx::tc_commit_pair(drain);
      else
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
      uint32_t se = 0, sph = 0;  // scale entry and its slot's phase
      bool ok = true;
      for (WorkIter wk(p, unit_first); ok && wk.valid; wk.next(p)) {
        int mu, nt;
        unit_coords(p, wk.u, mu, nt);
        const int mt = mu * CM + rank;
        const int m0 = mt * kBM, n0 = nt * BN;
        const int nb_first = n0 / 128;
        const int nb_count = (n0 + BN - 1) / 128 - nb_first + 1;
        const int kb_close = wk.last(p) ? wk.kb1 - 1 : KB;
#pragma unroll 1
        for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
          const uint32_t slot = se / kScaleGroup, sub = se % kScaleGroup;
          if (sub == 0) {
            bool w = wait_bar(&sempty[slot], sph ^ 1, abort_flag, kErrScales);
            if (!__all_sync(0xFFFFFFFFu, w)) { ok = false; break; }
          }
          // Asynchronous 4-byte copies (zero-filled outside the matrix) that
          // complete on sfull[slot]: the loader never waits for memory, so it
          // runs up to kScaleEntries K-groups ahead of the promotion warps.
          float* dst = sScale + se * L::kScaleFloats;
#pragma unroll
          for (int i = 0; i < kBM / 32; ++i) {
            const int r = lane + 32 * i, m = m0 + r;
            const bool v = m < p.M;
            ptx::cp_async_4(dst + r, v ? p.sa + (size_t)kb * p.M + m : p.sa, v);
          }
          float* dstb = dst + kBM;
          if (B_TILE) {
#pragma unroll
            for (int i = 0; i < BN / 32; ++i) {
              const int cidx = lane + 32 * i, n = n0 + cidx;
              const bool v = n < p.N;
              ptx::cp_async_4(dstb + cidx, v ? p.sb + (size_t)kb * p.N + n : p.sb, v);
            }
          } else if (lane < nb_count) {
            const int nb = nb_first + lane;
            const bool v = nb * 128 < p.N;
            ptx::cp_async_4(dstb + lane, v ? p.sb + (size_t)nb * KB + kb : p.sb, v);
          }
          // the slot is complete after its last K-group (or the CTA's last)
          if (sub == kScaleGroup - 1 || kb == kb_close) {
            ptx::cp_async_arrive_noinc(&sfull[slot]);
            se = (slot + 1) * kScaleGroup;
            if (se == kScaleEntries) {
              se = 0;
              sph ^= 1;
            }
          } else {
            ++se;
          }
        }
      }
      // no copy may still be in flight into shared memory when the CTA exits
      ptx::cp_async_wait_all();
    }
  }
  } else {
    // ------------------------------------------------- promotion + epilogue
    if constexpr (L::kRegSplit) ptx::regs_inc<L::kPromoRegs>();
    const int w = warp - kFirstPromoWarp;
    const int lg = warp & 3;       // TMEM lane group this warp may access
    const int ch = w >> 2;         // which kCols-wide column range
    const int row = lg * 32 + lane;
    const int col0 = ch * kCols;
    const uint32_t t_lane = (uint32_t)(lg * 32) << 16;
    uint32_t kt = 0;
    uint32_t se = 0, sph = 0;  // scale entry (0 .. kScaleEntries-1) and its slot's phase
    bool ok = true;
    for (WorkIter wk(p, unit_first); ok && wk.valid; wk.next(p)) {
      const int u = wk.u;
      int mu, nt;
      unit_coords(p, u, mu, nt);
      const int mt = mu * CM + rank;
      const int m0 = mt * kBM, n0 = nt * BN;
      float acc[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;

      if (PROMOTE) {
        using PS = PromoSteps<kCols>;
        constexpr int kS = PS::kSteps;
        static_assert(kS <= 4, "steps");
        // Block scales: the first column of this warp's range that lies in
        // the next 128-column block (kCols when there is none).
        // When the tile width and the warp's column range are whole 128-column
        // blocks (the 256-wide pair with 8 promotion warps), the range lies
        // in one block: one factor per K-group.
        constexpr bool kOneBlock = B_TILE || (BN % 128 == 0 && kCols % 128 == 0);
        const int a_split =
            kOneBlock ? kCols : ((n0 + col0) / 128 + 1) * 128 - (n0 + col0);
        const int nb_lo = (n0 + col0) / 128 - n0 / 128;
        // this K-group's row scale and block factors, from its scale slot
        auto read_scales = [&](const float* sc, float& sa_o, float& lo_o, float& hi_o) {
          sa_o = sc[row];
          lo_o = hi_o = 0.0f;
          if (!B_TILE) {
            lo_o = __fmul_rn(sa_o, sc[kBM + nb_lo]);
            hi_o = (!kOneBlock && a_split < kCols) ? __fmul_rn(sa_o, sc[kBM + nb_lo + 1]) : lo_o;
          }
        };
        uint32_t v[2][32];
        // the CTA's last K-group closes its scale slot early
        const int kb_close = wk.last(p) ? wk.kb1 - 1 : KB;
        // the next K-group's partial seen complete by a non-blocking test
        // issued during this K-group's last FMAs (double-buffered steps, tile
        // B scales: there the promotion is slower than the MMAs and the next
        // partial is nearly always ready; with block scales the early test
        // mostly fails and costs 8%)
        bool pre_full = false;
#pragma unroll 1
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++kt) {
          const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
          const uint32_t slot = se / kScaleGroup, sub = se % kScaleGroup;
          const float* sc = sScale + se * L::kScaleFloats;
          const float* scb = sc + kBM;
          const uint32_t tcur = tmem_base + t_lane + buf * L::kTmemStride + col0;
          float sa_r, f_lo, f_hi;
          if (sub == 0) {
            bool w1 = wait_bar(&sfull[slot], sph, abort_flag, kErrPromo);
            if (!__all_sync(0xFFFFFFFFu, w1)) { ok = false; break; }
          }
          read_scales(sc, sa_r, f_lo, f_hi);
          if (!B_TILE || !__all_sync(0xFFFFFFFFu, pre_full)) {
            bool w2 = wait_bar(&tfull[buf], tph, abort_flag, kErrPromo);
            if (!__all_sync(0xFFFFFFFFu, w2)) { ok = false; break; }
          }
          pre_full = false;
          ptx::tc_fence_after();
          if constexpr (L::kLoadAll) {
            // The whole partial of this warp in one round of loads; the
            // buffer goes back to the MMA issuer before the FMAs.
            uint32_t va[kCols];
            ptx::tmem_ld_cols<kCols>(tcur, va);
            ptx::tmem_ld_wait();
            reg_fence<kCols>(va);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) release_tmem<PAIR>(&tempty[buf]);
#pragma unroll
            for (int c = 0; c < kCols; c += 16)
              promote_step<16, 0, B_TILE>(acc + c, va + c, sa_r, scb, col0 + c, f_lo, f_hi,
                                          a_split - c);
          } else if constexpr (L::kSingleBuf) {
            // One register buffer: load a step, wait, (after the last load)
            // hand the buffer back, then the step's FMAs.
            uint32_t* v1 = v[0];
#define FP8BS_STEP1(S)                                                                    \
  if constexpr (S < kS) {                                                                 \
    tmem_ld_step<PS::width(S)>(tcur + 32 * (S), v1);                                      \
    ptx::tmem_ld_wait();                                                                  \
    reg_fence<PS::width(S)>(v1);                                                          \
    if constexpr (S + 1 == kS) {                                                          \
      ptx::tc_fence_before();                                                             \
      __syncwarp();                                                                       \
      if (lane == 0) release_tmem<PAIR>(&tempty[buf]);                                    \
    }                                                                                     \
    promote_step<PS::width(S), 32 * (S), B_TILE, 16>(acc, v1, sa_r, scb, col0, f_lo, f_hi, \
                                                     a_split);                            \
  }
            FP8BS_STEP1(0)
            FP8BS_STEP1(1)
            FP8BS_STEP1(2)
            FP8BS_STEP1(3)
#undef FP8BS_STEP1
          } else {
            // Double-buffered steps: the load of step s+1 is issued right
            // after step s's data has arrived and before step s's FMAs
            // (tcgen05.wait::ld waits for all of this thread's loads, so one
            // step is in flight at a time).
            tmem_ld_step<PS::width(0)>(tcur, v[0]);
#define FP8BS_STEP(S)                                                                     \
  if constexpr (S < kS) {                                                                 \
    ptx::tmem_ld_wait();                                                                  \
    reg_fence<PS::width(S)>(v[S & 1]);                                                    \
    if constexpr (S + 1 < kS) {                                                           \
      tmem_ld_step<PS::width(S + 1)>(tcur + 32 * (S + 1), v[(S + 1) & 1]);                \
    } else {                                                                              \
      /* every TMEM read of this buffer is done: hand it back */                          \
      ptx::tc_fence_before();                                                             \
      __syncwarp();                                                                       \
      if (lane == 0) release_tmem<PAIR>(&tempty[buf]);                                    \
      if (B_TILE && kb + 1 < wk.kb1)                                                      \
        pre_full = ptx::mbar_test_wait(ptx::smem_addr(&tfull[(kt + 1) % TBUF]),           \
                                       ((kt + 1) / TBUF) & 1);                            \
    }                                                                                     \
    promote_step<PS::width(S), 32 * S, B_TILE>(acc, v[S & 1], sa_r, scb, col0, f_lo, f_hi, \
                                               a_split);                                  \
  }
            FP8BS_STEP(0)
            FP8BS_STEP(1)
            FP8BS_STEP(2)
            FP8BS_STEP(3)
#undef FP8BS_STEP
          }
          if (sub == kScaleGroup - 1 || kb == kb_close) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sempty[slot]);
            // the next K-group starts the next slot
            se = (slot + 1) * kScaleGroup;
            if (se == kScaleEntries) {
              se = 0;
              sph ^= 1;
            }
          } else {
            ++se;
          }
        }
        if (!ok) break;
      } else {
        const uint32_t buf = kt % TBUF, tph = (kt / TBUF) & 1;
        bool w2 = wait_bar(&tfull[buf], tph, abort_flag, kErrPromo);
        if (!__all_sync(0xFFFFFFFFu, w2)) { ok = false; break; }
        ptx::tc_fence_after();
        const int m = m0 + row;
        const float sa_r = (m < p.M) ? __ldg(p.sa + m) : 0.0f;  // K-group 0
        const uint32_t tbase = tmem_base + t_lane + buf * L::kTmemStride + col0;
#pragma unroll
        for (int c0 = 0; c0 < kCols / 16; ++c0) {
          uint32_t v[16];
          ptx::tmem_ld_32x32b_x16(tbase + c0 * 16, v);
          ptx::tmem_ld_wait();
          reg_fence<16>(v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = n0 + col0 + c0 * 16 + j;
            float sbv = 0.0f;
            if (n < p.N) sbv = B_TILE ? __ldg(p.sb + n) : __ldg(p.sb + (size_t)(n / 128) * p.KB);
            acc[c0 * 16 + j] = __fmul_rn(__uint_as_float(v[j]), __fmul_rn(sa_r, sbv));
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) release_tmem<PAIR>(&tempty[buf]);
        ++kt;
      }
      if (!ok) break;

      if (PROMOTE && OUT != kOutE4m3 && (wk.kb0 != 0 || wk.kb1 != KB)) {
        // A stream-K unit split over CTA groups g_first .. g_last.  Every
        // share goes to the workspace (this warp's 32 rows x kCols, laid out
        // so that each float4 store of the warp covers 512 contiguous bytes),
        // then an arrival counter per (unit, CTA, warp) picks the last
        // arriver, which sums the shares in K order and writes the tile.
        const int tsk = u - p.sk_begin;
        const int t_it0 = tsk * KB;
        const int g_first = sk_owner(p, t_it0), g_last = sk_owner(p, t_it0 + KB - 1);
        const size_t chunk = (size_t)32 * kCols / 4;  // float4s per warp share
        auto share = [&](int g) {
          return reinterpret_cast<float4*>(p.ws) +
                 (((size_t)sk_slot(p, g, u) * CM + rank) * kPromoWarps + w) * chunk;
        };
        // one base address per share, each float4 at an immediate offset
        const float4* mine = share(unit_first) + lane;
        share_store<kCols>(mine, acc);
        __threadfence();
        __syncwarp();
        unsigned int* cnt = p.ws_cnt + ((size_t)tsk * CM + rank) * kPromoWarps + w;
        unsigned int ticket = 0;
        if (lane == 0) ticket = atomicAdd(cnt, 1u);
        ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
        if ((int)ticket != g_last - g_first) continue;  // another group finishes the unit
        __threadfence();
        // every share, this group's included, read back in K order: acc =
        // ((share_first + share_next) + ...) whichever group arrives last
        share_sum<kCols>(acc, [&](int g) { return share(g) + lane; }, g_first, g_last);
        if (lane == 0) *cnt = 0u;  // ready for the next launch
      }

      // ---- epilogue: registers -> global (bf16 RNE or fp32)
      constexpr bool kTmaOut = L::kEpiTma && OUT != kOutE4m3;
      if constexpr (kTmaOut) {
        // Through the warp's 4 KB staging tile and one tensor store per
        // chunk of columns; the store clips rows and columns outside C, and
        // the warp goes on to the next unit while the stores drain.  Chunks
        // of 128 bytes per row (32 FP32 or 64 BF16 columns) when the warp's
        // columns are whole such chunks, staged in the 128-byte-swizzled
        // layout of the tensor map (16-byte chunk c of row r at c ^ (r % 8),
        // so each quarter warp's writes hit distinct banks); otherwise chunks
        // of 16 columns, unswizzled rows of 64 or 32 bytes.
        constexpr int kElt = OUT == kOutF32 ? 4 : 2;
        constexpr bool kWide = kCols % (128 / kElt) == 0;
        constexpr int kChunk = kWide ? 128 / kElt : 16;  // columns per store
        constexpr int kRowBytes = kChunk * kElt;
        uint8_t* ebuf = smem + L::kOffEpi + w * 4096;
#pragma unroll
        for (int j0 = 0; j0 < kCols; j0 += kChunk) {
          if (lane == 0) ptx::bulk_wait_read_all();  // the last store has read the tile
          __syncwarp();
#pragma unroll
          for (int c = 0; c < kRowBytes / 16; ++c) {
            uint4 v;
            if constexpr (OUT == kOutF32) {
              const int j = j0 + 4 * c;
              v = make_uint4(__float_as_uint(acc[j]), __float_as_uint(acc[j + 1]),
                             __float_as_uint(acc[j + 2]), __float_as_uint(acc[j + 3]));
            } else {
              const int j = j0 + 8 * c;
              __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[j], acc[j + 1]);
              __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[j + 2], acc[j + 3]);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[j + 4], acc[j + 5]);
              __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[j + 6], acc[j + 7]);
              v = make_uint4(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                             *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
            }
            const int pos = kWide ? (c ^ (lane & 7)) : c;
            *reinterpret_cast<uint4*>(ebuf + lane * kRowBytes + (pos << 4)) = v;
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmap_c, ebuf, n0 + col0 + j0, m0 + lg * 32);
            ptx::bulk_commit();
          }
        }
        continue;
      }
      static_assert(kTmaOut || OUT == kOutE4m3, "FP32 and BF16 outputs use tensor stores");
      if constexpr (OUT == kOutE4m3) {
        const int m = m0 + row;
        if (m < p.M) {
          // One 1x128 group of the output row per thread: the warp's
          // kCols = 128 columns start on a multiple of 128.  Same rule as the
          // activation quantizer on FP32 values: s = fl32(amax / 448), codes
          // of fl32(x / s) (two correction steps: x is a full FP32 value).
          static_assert(kCols == 128, "one 1x128 group per promotion thread");
          const int n = n0 + col0;
          if (n < p.N) {
            float amax = 0.0f;  // NaN if the group holds a NaN
#pragma unroll
            for (int j2 = 0; j2 < kCols; ++j2) amax = fmax_abs_nan(amax, acc[j2]);
            float mn = amax;
            if (amax != amax) {  // rare: recount ignoring NaN
              mn = 0.0f;
#pragma unroll
              for (int j2 = 0; j2 < kCols; ++j2) mn = fmaxf(mn, fabsf(acc[j2]));
            }
            const GroupScale g =
                make_scale(__float_as_uint(mn), !(amax < __uint_as_float(0x7F800000u)), false);
            uint8_t* crow = static_cast<uint8_t*>(p.c) + (size_t)m * p.N + n;
#pragma unroll
            for (int j2 = 0; j2 < kCols; j2 += 16) {
              uint4 o;
              o.x = codes_f32x4(acc[j2], acc[j2 + 1], acc[j2 + 2], acc[j2 + 3], g);
              o.y = codes_f32x4(acc[j2 + 4], acc[j2 + 5], acc[j2 + 6], acc[j2 + 7], g);
              o.z = codes_f32x4(acc[j2 + 8], acc[j2 + 9], acc[j2 + 10], acc[j2 + 11], g);
              o.w = codes_f32x4(acc[j2 + 12], acc[j2 + 13], acc[j2 + 14], acc[j2 + 15], g);
              *reinterpret_cast<uint4*>(crow + j2) = o;
            }
            p.c_scales[(size_t)(n / 128) * p.M + m] = g.s;
          }
        }
      }
    }
    // this warp's output tensor stores have completed before the CTA exits
    if (lane == 0) ptx::bulk_wait_all();
  }

  // ---- teardown: all roles done (or aborted); free TMEM
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) {
    // Neither CTA leaves (or frees TMEM the pair's MMAs write) while the
    // other may still touch it.  Copies land only in the issuing CTA's own
    // shared memory; the follower's copies complete on the leader's full
    // barriers, which the leader's producer has drained above, and the
    // leader's MMAs (which read both CTAs' shared memory) were drained by
    // its MMA issuer, before either CTA arrives here.
    ptx::cluster_sync();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR)
      ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

// Row-major uint8 matrix [rows][cols] (cols contiguous), box of box_rows x
// 128 bytes with the 128-byte swizzle; out-of-range rows read as zero.
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  return make_tmap_2d(map, base, 1, rows, cols, 128, box_rows, true);
}

constexpr int kMaxDevices = 64;

int num_sms_current_device() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// Per-device, per-kernel launch facts, computed on first use: the
// shared-memory attribute is set, the register split is checked against
// what the compiled kernel is launched with, and for clusters the number of
// clusters that fit on the device at once.
// Host threads may launch concurrently: the first to arrive computes the
// facts under the mutex and publishes them with a release store.
struct KernelInfo {
  std::atomic<bool> ready{false};
  std::mutex mu;
  cudaError_t err = cudaSuccess;
  int max_ctas = 0;  // persistent grid size (a multiple of CM)
};

// Stream-K's cost in waves beyond the work itself, fitted to timings of
// 128 x 256 tiles: split over every CTA, 448 tiles (3.03 waves) ran like
// 3.56 waves and 896 tiles (6.05 waves) like 6.61.
constexpr double kSkCostWaves = 0.55;

// Whether spreading the last waves over every CTA group beats whole units:
// the last wave of `units` whole units on `groups` groups leaves them idle
// for more than stream-K's cost.
inline bool sk_worth(int64_t units, int64_t groups) {
  if (groups <= 0 || units <= 0) return false;
  const int64_t waves = (units + groups - 1) / groups;
  return (double)waves - (double)units / groups > kSkCostWaves;
}

template <int BN, bool PAIR, int PW, bool PROMOTE, int OUT, bool B_TILE>
cudaError_t launch_variant(const GemmArgs& g, cudaStream_t stream) {
  using L = Cfg<BN, PAIR, PW>;
  constexpr int CM = L::CM;
  constexpr int kThreads = L::kThreads;
  auto kern = gemm_kernel<BN, PAIR, PW, PROMOTE, OUT, B_TILE>;
  static KernelInfo info[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  KernelInfo& ki = info[dev];
  if (!ki.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(ki.mu);
    if (!ki.ready.load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
      if (e == cudaSuccess && L::kRegSplit) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        // setmaxnreg.inc waits until the registers it asks for are free: a
        // split larger than the launch's allocation would never proceed.
        if (e == cudaSuccess && fa.numRegs * kThreads < L::kSplitRegsNeeded)
          e = cudaErrorInvalidConfiguration;
      }
      int ctas = num_sms_current_device();
      if (e == cudaSuccess && CM > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CM * 64);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = L::kAlloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CM;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e == cudaSuccess && clusters < 1) e = cudaErrorInvalidConfiguration;
        ctas = clusters * CM;
      }
      ki.err = e;
      ki.max_ctas = ctas;
      ki.ready.store(true, std::memory_order_release);
    }
  }
  if (ki.err != cudaSuccess) return ki.err;

  // Stream-K plan.  When the last wave of whole units would leave the CTA
  // groups idle for more than sk_worth's share of a wave (e.g. 16 pair
  // tiles on 74 pairs, or 448 one-CTA tiles on 148 CTAs: 3.03 waves), the
  // units of the last two waves (all of them, below two waves) have their
  // K-groups spread evenly over every group.  Below that, the shares'
  // hand-off through the workspace costs more than the idle groups
  // (measured: 128 tiles on 74 pairs, 1.73 waves, ran 12% slower split).
  // Workspace:
  // two FP32 shares of a CTA's 128 x BN accumulator per group (the partial
  // first and last segments of its share), then one arrival counter per
  // stream-K unit, CTA and promotion warp.
  const int64_t m_units = ((g.M + kBM - 1) / kBM + CM - 1) / CM;
  const int64_t all_units = m_units * ((g.N + BN - 1) / BN);
  const int64_t groups = ki.max_ctas / CM;
  int64_t sk_begin = all_units;
  size_t ws_shares = 0, ws_need = 0;
  if (PROMOTE && OUT != kOutE4m3 && (g.ws != nullptr || g.ws_need != nullptr) && groups > 0) {
    // (the stream-K iteration count must fit an int)
    const int64_t sk_units_max = all_units / groups >= 1 ? all_units % groups + groups : all_units;
    if (sk_worth(all_units, groups) && sk_units_max * (g.K / kBK) < (int64_t(1) << 31)) {
      sk_begin = all_units / groups >= 1 ? (all_units / groups - 1) * groups : 0;
      ws_shares = (size_t)2 * groups * CM * kBM * BN * sizeof(float);
      ws_need = ws_shares + (size_t)(all_units - sk_begin) * CM * PW * sizeof(unsigned int);
    }
  }
  if (g.ws_need != nullptr) {
    *g.ws_need = ws_need;
    return cudaSuccess;
  }
  if (ws_need > g.ws_bytes) return cudaErrorInvalidValue;

  CUtensorMap ta, tb, tc = {};
  if (!make_tmap(&ta, g.a, g.M, g.K, kBM) || !make_tmap(&tb, g.b, g.N, g.K, L::kBH))
    return cudaErrorInvalidValue;
  // C for the tensor-store epilogue: 32 rows x 128 bytes per box (swizzled)
  // when the warps' columns are whole 128-byte chunks, else 32 rows x 16
  // columns (unswizzled)
  if (L::kEpiTma && OUT != kOutE4m3) {
    const int elt = OUT == kOutF32 ? 4 : 2;
    const bool wide = L::kCols % (128 / elt) == 0;
    if (!make_tmap_2d(&tc, g.c, elt, g.M, g.N, wide ? 128 / elt : 16, 32, wide))
      return cudaErrorInvalidValue;
  }
  Params p;
  p.sa = g.sa;
  p.sb = g.sb;
  p.c = g.c;
  p.c_scales = g.c_scales;
  p.M = (int)g.M;
  p.N = (int)g.N;
  p.K = (int)g.K;
  p.KB = (int)(g.K / kBK);
  const int m_tiles = (int)((g.M + kBM - 1) / kBM);
  p.num_m_units = (m_tiles + CM - 1) / CM;
  const int n_tiles = (int)((g.N + BN - 1) / BN);
  p.num_units = p.num_m_units * n_tiles;
  p.num_n_units = n_tiles;
  p.skip_iter = g.skip_iter;
  int units = ki.max_ctas / CM;
  if (units > p.num_units && ws_need == 0) units = p.num_units;
  p.num_groups = units;
  p.sk_begin = (int)sk_begin;
  p.sk_iters = (int)((all_units - sk_begin) * p.KB);
  p.sk_q = p.sk_iters / units;
  p.sk_r = p.sk_iters % units;
  p.ws = nullptr;
  p.ws_cnt = nullptr;
  if (ws_need > 0) {
    p.ws = static_cast<float*>(g.ws);
    p.ws_cnt = reinterpret_cast<unsigned int*>(static_cast<char*>(g.ws) + ws_shares);
    // the counters start every launch at zero (a launch that timed out may
    // have left some behind)
    e = cudaMemsetAsync(p.ws_cnt, 0, ws_need - ws_shares, stream);
    if (e != cudaSuccess) return e;
  }
  // Group size: the units in flight (about `units`) cover group_m unit rows
  // and units / group_m tile columns; A bytes grow with the first, B bytes
  // with the second, and group_m = sqrt(units * BN / unit rows) balances them.
  {
    int gm = (int)(sqrtf((float)units * (float)BN / (float)(CM * kBM)) + 0.5f);
    if (gm < 1) gm = 1;
    if (gm > p.num_m_units) gm = p.num_m_units;
    p.group_m = gm;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * CM);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (CM > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = CM;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Tile shape per problem.  Each candidate's cost is the number of waves it
// needs times its tile width over a relative efficiency (measured per shape
// on B300: the 256-row CTA pairs read half the B operand per MAC from shared
// memory that one-CTA tiles do, and wider tiles read less A per MAC); the
// cheapest wins.
enum TileShape {
  kTile128x128 = 0,
  kTile128x256 = 1,
  kTile256x128Pair = 2,
  kTile256x160Pair = 3,
  kTile256x192Pair = 4,
  kTile256x224Pair = 5,
  kTile256x256Pair = 6,
  kTile256x192PairW12 = 7,
  kTile256x256PairW16 = 8,
  kTile256x192PairW16 = 9,
  kTile256x128PairW16 = 10,
};

TileShape choose_tile(int64_t M, int64_t N, int sms, bool streamk) {
  struct Cand {
    TileShape s;
    int bm, bn;
    double eff;
  };
  // Efficiencies fitted to interleaved timings of every shape on the dense,
  // MoE, Dgrad, Wgrad and stress workloads (relative per-wave times at equal
  // waves).  The one-CTA 128 x 256 tile has the 256 x 256 pair's waves (twice
  // the units on twice the slots) and measured 1-4% faster than it.
  const Cand cands[] = {{kTile128x256, 128, 256, 1.02},     {kTile256x256Pair, 256, 256, 1.0},
                        {kTile256x224Pair, 256, 224, 0.89}, {kTile256x192Pair, 256, 192, 0.82},
                        {kTile256x160Pair, 256, 160, 0.82}, {kTile256x128Pair, 256, 128, 0.63},
                        {kTile128x128, 128, 128, 0.65}};
  TileShape best = kTile128x128;
  double best_cost = 1e300;
  for (const Cand& c : cands) {
    const int64_t units = ((M + c.bm - 1) / c.bm) * ((N + c.bn - 1) / c.bn);
    const int64_t slots = sms / (c.bm / kBM);
    const int64_t waves = (units + slots - 1) / slots;
    // with stream-K (when the plan would split this shape) the work counts
    // in fractional waves plus the hand-off's cost
    const double w = streamk && sk_worth(units, slots) ? (double)units / slots + kSkCostWaves
                                                       : (double)waves;
    const double cost = w * c.bn / c.eff;
    if (cost < best_cost) {
      best_cost = cost;
      best = c.s;
    }
  }
  return best;
}

template <bool PROMOTE, int OUT, bool B_TILE>
cudaError_t launch_shape(const GemmArgs& g, cudaStream_t stream) {
  // E4M3 output needs each promotion thread to own one whole 1x128 group of
  // an output row: the 256 x 256 pair (two 128-column halves per row)
  if constexpr (OUT == kOutE4m3) {
    return launch_variant<256, true, 8, PROMOTE, OUT, B_TILE>(g, stream);
  } else {
    int shape = g.tile;
    if (shape < 0) {
      // stream-K calls (a workspace given or asked for) weigh each shape
      // with the stream-K plan it would get
      shape = choose_tile(g.M, g.N, num_sms_current_device(),
                          PROMOTE && (g.ws != nullptr || g.ws_need != nullptr));
      // the un-promoted variant runs at the tensor pipe's rate, where the
      // pair's halved B reads from shared memory matter: the 256 x 256 pair
      // in place of the one-CTA 128 x 256 tile (same waves)
      if (!PROMOTE && shape == kTile128x256) shape = kTile256x256Pair;
    }
    switch (shape) {
      case kTile256x192PairW12:
        return launch_variant<192, true, 12, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x256PairW16:
        return launch_variant<256, true, 16, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x192PairW16:
        return launch_variant<192, true, 16, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x128PairW16:
        return launch_variant<128, true, 16, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x128Pair:
        return launch_variant<128, true, 8, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x160Pair:
        return launch_variant<160, true, 8, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x192Pair:
        return launch_variant<192, true, 8, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x224Pair:
        return launch_variant<224, true, 8, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile256x256Pair:
        return launch_variant<256, true, 8, PROMOTE, OUT, B_TILE>(g, stream);
      case kTile128x256:
        return launch_variant<256, false, 8, PROMOTE, OUT, B_TILE>(g, stream);
      default:
        return launch_variant<128, false, 8, PROMOTE, OUT, B_TILE>(g, stream);
    }
  }
}

template <bool PROMOTE, int OUT>
cudaError_t launch_bt(const GemmArgs& g, cudaStream_t stream) {
  return g.b_tile ? launch_shape<PROMOTE, OUT, true>(g, stream)
                  : launch_shape<PROMOTE, OUT, false>(g, stream);
}

template <bool PROMOTE>
cudaError_t launch_out(const GemmArgs& g, cudaStream_t stream) {
  switch (g.out) {
    case kOutBf16:
      return launch_bt<PROMOTE, kOutBf16>(g, stream);
    case kOutE4m3:
      if constexpr (PROMOTE) return launch_bt<PROMOTE, kOutE4m3>(g, stream);
      return cudaErrorInvalidValue;
    default:
      return launch_bt<PROMOTE, kOutF32>(g, stream);
  }
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  return g.promote ? launch_out<true>(g, stream) : launch_out<false>(g, stream);
}

// Moves the error word into *dst and clears it in one atomic step, in
// stream order: an error set by any kernel on the device is taken by exactly
// one query.
__global__ void take_gemm_error_kernel(unsigned int* dst) {
  *dst = atomicExch(&g_device_error, 0u);
}

cudaError_t enqueue_take_gemm_error(unsigned int* dst, cudaStream_t stream) {
  take_gemm_error_kernel<<<1, 1, 0, stream>>>(dst);
  return cudaGetLastError();
}

}  // namespace fp8bs
