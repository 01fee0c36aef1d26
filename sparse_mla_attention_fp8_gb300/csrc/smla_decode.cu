// FP8 sparse MLA decode on sm_103a, reading the 656-byte cache rows as stored.
//
// What is computed (vLLM flashmla_sparse.py: the "FP8 with scale" row format
// in the module docstring, FlashMLASparseImpl.forward and its FP8 decode
// kernel call): for each query token t and each of its H heads,
//   s_j = softmax_scale * <q[t,h,:], K_j>, K_j = [e4m3(c) * scale_j[c/128] for
//         c < 512] ++ RoPE_j (64 bf16),
//   out = sum_j softmax(s)_j * K_j[0:512],  lse = log sum_j exp(s_j),
// over the token's top-k rows (translated through the paged block table);
// invalid rows are masked, a token without valid rows gets out = 0, lse = -inf.
//
// Design: the tensor cores read the cache codes as stored, with no
// dequantization pass.
//  * Transport: TMA tile::gather4 copies straight into the operand tiles,
//    four rows per instruction: the 512 e4m3 codes as four K-major panels with
//    the 128-byte swizzle (64 rows x 128 bytes each), the 64 bf16 RoPE values
//    as a fifth panel; the four float32 scales of a row go beside them as one
//    16-byte cp.async, which keeps these small copies out of the TMA queue.
//    Invalid rows are gathered at row -1, which the TMA zero-fills (the scale
//    copy writes zeros).  Four loader warps, one per
//    16-row quarter of every tile, each lane issuing one copy: the cost of
//    issuing copies falls on the issuing warp, so it is spread.  Four operand
//    tiles, so that the loads of the next tiles are in flight while one is
//    in use.
//  * Q is split once per (token, 16-head group) into two e4m3 terms,
//    q * 2^s_hg = hi + lo (s_hg a power of two per head and 128-column scale
//    group g putting the group's max |q| near 448), exact for all but
//    components far below their group's largest; hi and lo are the two halves
//    of an N = 32 operand.  QK^T for each scale group g is one kind::f8f6f4
//    product E_g [Q_hi Q_lo]^T (M = 64 rows, N = 32, K = 128 codes), the RoPE
//    part a bf16 product; the softmax combines
//    s = sum_g scale_g 2^-s_hg (S_g,hi + S_g,lo) + S_rope in fp32.
//  * P.V for value chunk q (= scale group q) is one kind::f8f6f4 product
//    O_q^T += E_q^T P'_q with the same code panel read MN-major and
//    P'_q = 2^7 p * scale_q / R_q split into e4m3 hi + lo (R_q a running
//    power-of-two bound of the group's scales).  The running max of a head is
//    refreshed (to 2^0.75 above the tile's maximum) only when a tile's maximum
//    exceeds it by more than 2^1.75, so p <= 2^1.75 and P' < 430 stays at the
//    top of the e4m3 range (max 448), where hi + lo carries 8 significant
//    bits.  O is rescaled in tensor memory when R_q or a running max changes;
//    the slack and overshoot keep that to a few tiles per unit.  P' is
//    double-buffered.
//  * Heads live in "S column" order throughout: column n of S, of P' and of O
//    holds head pi(n) = 4 ((n & 7) >> 1) + (n & 1) + 2 (n >> 3); only the
//    output stores translate.
//  * Warp roles: softmax / epilogue (8 warps: two per TMEM lane quarter, one
//    per half of the 16 head columns), tensor-core issuer (1 thread), index
//    translation (1 warp), loaders (4 warps), Q preparation (2 warps).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "smla_combine.cuh"
#include "smla_common.cuh"
#include "smla_kernels.h"

namespace smla {

namespace {

constexpr uint32_t kFullMask = 0xffffffffu;

// Optional per-tile timeline for performance work: with SMLA_TRACE defined,
// roles record %globaltimer at their hand-off points into g_smla_trace_fp8
// (set by the host through smla_trace_set_fp8).  Compiled out otherwise.
#ifdef SMLA_TRACE
__device__ unsigned long long* g_smla_trace_fp8 = nullptr;
constexpr int kTraceTiles = 64, kTraceEvents = 19;
enum { kEvIdx = 0, kEvRawLanded = 1, kEvOpFull = 2, kEvQk = 3, kEvSoftStart = 4, kEvSoftDone = 5, kEvPv = 6,
       kEvQReady = 7, kEvRawFull = 8, kEvOpEmpty = 9, kEvIssue = 10, kEvSoftLogits = 11, kEvSoftBar = 12,
       kEvSoftPWait = 13, kEvQkSeen = 14, kEvPvSeen = 15, kEvRawFullH1 = 16,
       kEvRawLandedH1 = 17, kEvIssueH1 = 18 };
#define SMLA_TRACE_SET(tl, ev)                                                                                  \
  do {                                                                                                          \
    if (g_smla_trace_fp8 && (tl) < kTraceTiles)                                                                  \
      g_smla_trace_fp8[((size_t)blockIdx.x * kTraceTiles + (tl)) * kTraceEvents + (ev)] = globaltimer_ns();    \
  } while (0)
// Cycle counters of the softmax sections (thread 0), stored after the per-tile events.
#define SMLA_CLK_DECL unsigned clk_acc[16] = {0}, clk_prev = (unsigned)clock()
#define SMLA_CLK_START() SMLA_CLK_MARK(13)
#define SMLA_CLK_MARK(i)                   \
  do {                                     \
    const unsigned now_ = (unsigned)clock(); \
    clk_acc[(i)] += now_ - clk_prev;       \
    clk_prev = now_;                       \
  } while (0)
#define SMLA_CLK_STORE()                                                                                        \
  do {                                                                                                          \
    if (g_smla_trace_fp8 && tid == 0)                                                                           \
      for (int i_ = 0; i_ < 16; ++i_)                                                                           \
        g_smla_trace_fp8[(size_t)gridDim.x * kTraceTiles * kTraceEvents + blockIdx.x * 16 + i_] = clk_acc[i_]; \
  } while (0)
#else
#define SMLA_TRACE_SET(tl, ev) ((void)0)
#define SMLA_CLK_DECL
#define SMLA_CLK_START() ((void)0)
#define SMLA_CLK_MARK(i) ((void)0)
#define SMLA_CLK_STORE() ((void)0)
#endif

constexpr int HG = 16;                 // heads per CTA work unit
constexpr int kRows = 64;              // top-k rows per tile
constexpr int kLoaders = 4;            // loader warps: loader lw gathers rows 16 lw .. 16 lw + 15 of every tile
constexpr int kOpBufs = 4;             // operand tiles
constexpr float kMaxSlack = 1.75f;     // log2 growth of a head's max tolerated before rescaling O (p <= 2^1.75)
constexpr float kMaxOvershoot = 0.75f; // a refreshed running max is set this far above the tile max
constexpr float kPScale = 128.0f;      // P' = kPScale * p * scale / R  <=  128 * 2^1.75 < 430 (e4m3 max 448)
constexpr float kPScaleInv = 1.0f / 128.0f;

// ---- shared memory layout (offsets from a 1024-byte aligned base)
constexpr int kPanel = kRows * 128;                   // 8 KB: 64 rows x 128 bytes
constexpr int kOpRope = 4 * kPanel;                   // RoPE panel after the 4 code panels
constexpr int kOpScale = 5 * kPanel;                  // scales: 16 groups of 4 rows x 16 bytes, 128 bytes apart
constexpr int kOpBuf = 5 * kPanel + (kRows / 4) * 128;  // 43008
constexpr int kQPanel = 32 * 128;                     // 32 operand rows (hi, lo) x 128 codes
constexpr int kQRope = 4 * kQPanel;                   // 16 rows x 64 bf16
constexpr int kQBuf = 4 * kQPanel + HG * 128;         // 18432
constexpr int kPGroup = kRows * 32;                   // P'_q: 64 rows x 32 codes
constexpr int kPBuf = 4 * kPGroup;                    // 8192
constexpr int kOffOp = 0;
constexpr int kOffQ = kOffOp + kOpBufs * kOpBuf;
constexpr int kOffP = kOffQ + kQBuf;
constexpr int kPBufs = 3;                                           // P' buffers
constexpr int kOffSlots = kOffP + kPBufs * kPBuf;                   // int32 [4][64]
constexpr int kOffValid = kOffSlots + 4 * kRows * 4;                // uint8 [4][64]
constexpr int kOffPre = kOffValid + kOpBufs * kRows;                // float [4][4 groups][16 columns] inverse Q prescales
constexpr int kOffRedMax = kOffPre + 4 * 4 * HG * 4;                    // float [2][4 quarters][16 columns]
constexpr int kOffRedSc = kOffRedMax + 2 * 4 * HG * 4;              // float [2][2 halves][4 quarters][4]
constexpr int kOffRedSum = kOffRedSc + 2 * 2 * 4 * 4 * 4;           // float [4 quarters][16 columns]
constexpr int kOffBar = kOffRedSum + 4 * HG * 4;
enum {
  kBarOpFull = 0, kBarOpEmpty = kBarOpFull + kOpBufs, kBarSFull = kBarOpEmpty + kOpBufs, kBarSFree = kBarSFull + 2,
  kBarPFull = kBarSFree + 2,
  kBarPvDone = kBarPFull + kPBufs, kBarIdxFull = kBarPvDone + kPBufs, kBarIdxEmpty = kBarIdxFull + 4,
  kBarQFull = kBarIdxEmpty + 4, kBarQEmpty = kBarQFull + 1, kBarOFree = kBarQEmpty + 1, kBarDrain = kBarOFree + 1,
  kNumBars = kBarDrain + 1
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kOpBuf % 1024 == 0, "operand alignment");
static_assert(kOffBar % 8 == 0, "barriers 8-byte aligned");
static_assert(kOffPre % 16 == 0 && kOffRedMax % 16 == 0 && kOffRedSc % 16 == 0 && kOffRedSum % 16 == 0, "float4");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// ---- tensor memory columns
constexpr int kSCols = 4 * 32 + HG;   // per S buffer: 4 groups x (hi, lo) x 16 heads + RoPE
constexpr int kOCol = 2 * kSCols;     // O^T: 4 chunks x (hi, lo) x 16 heads
constexpr int kTmemCols = 512;
static_assert(kOCol + 4 * 32 <= kTmemCols, "tensor memory budget");

// ---- warp roles (16 warps; 128 registers per thread).  Warp w runs on
// sub-partition w % 4: each sub-partition carries two softmax warps (one per
// head half), a loader and one more role.
constexpr int kSoftWarps = 8, kLoadWarp0 = 8, kMmaWarp = 12, kIndexWarp = 13, kQWarp0 = 14, kQWarps = 2;
constexpr int kNumWarps = 16;
constexpr int kThreads = 32 * kNumWarps;
static_assert(kLoadWarp0 + kLoaders == kMmaWarp && kQWarp0 + kQWarps == kNumWarps, "warp roles");

__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// 16-byte cp.async global -> shared (src_bytes = 0 writes zeros), and an
// arrival on an mbarrier once every earlier cp.async of this thread has
// landed (the barrier's count includes it).
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

struct Params {
  const __nv_bfloat16* q;
  const uint8_t* cache;
  const int32_t* indices;
  const int32_t* block_table;
  const int32_t* req_id;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int* status;
  float scale_log2;
  int T, H, K, R, MB;
  int64_t NB;
  int n_hg, nt;
  int64_t total;
  int G;
};

struct TileInfo {
  int u, kt, t, hg;
  bool seg_start, seg_end;
};

__device__ __forceinline__ TileInfo tile_info(const Params& p, int64_t x, int64_t xbeg, int64_t xend) {
  TileInfo ti;
  ti.u = (int)(x / p.nt);
  ti.kt = (int)(x - (int64_t)ti.u * p.nt);
  ti.t = ti.u / p.n_hg;
  ti.hg = ti.u - ti.t * p.n_hg;
  ti.seg_start = (x == xbeg) || (ti.kt == 0);
  ti.seg_end = (x == xend - 1) || (ti.kt == p.nt - 1);
  return ti;
}

__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// e4m3 pair (round to nearest even, saturating) of two floats: lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// decode an e4m3 pair (low byte first) to two floats (exact)
__device__ __forceinline__ float2 e4m3x2_decode(uint32_t pair16) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)pair16));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
// x -> (hi, lo) e4m3 codes with x = hi + lo wherever both are representable.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = e4m3x2(x0, x1);
  const float2 d = e4m3x2_decode(hi);
  lo = e4m3x2(x0 - d.x, x1 - d.y);
}

__device__ __forceinline__ float pow2_ceil(float x) {  // smallest power of two >= x (x > 0)
  const uint32_t u = __float_as_uint(x);
  const uint32_t e = u & 0x7F800000u;
  return __uint_as_float((u & 0x007FFFFFu) ? e + 0x00800000u : e);
}

// 1 / x for a power of two x in the normal range (exact).
__device__ __forceinline__ float rcp_pow2(float x) { return __uint_as_float(0x7F000000u - __float_as_uint(x)); }

__device__ __forceinline__ float ex2_approx(float x) {  // 2^x; 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Q operand row (and so S column) of head h: column n holds head pi(n) with
// pi(2c + e + 8d) = 4c + e + 2d, so that the 16x256b.x1 read of column half d
// gives thread c (lane % 4) the two adjacent columns 8d + 2c, 8d + 2c + 1.
__device__ __forceinline__ int q_row_of_head(int h) { return 2 * (h >> 2) + (h & 1) + 8 * ((h >> 1) & 1); }

// Head held by column n of S, P' and O (the inverse of q_row_of_head).
__device__ __forceinline__ int head_of_col(int n) { return 4 * ((n & 7) >> 1) + (n & 1) + 2 * (n >> 3); }

// Two floats -> e4m3 hi and lo pairs (low byte from x0), x ~ hi + lo; the
// split runs in f16x2 (11 significant bits, more than the 8 that hi + lo keep).
__device__ __forceinline__ void split2_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  uint32_t a, d, r;
  uint16_t t;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(a) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(t) : "r"(a));
  hi = t;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(t));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(d));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(t) : "r"(r));
  lo = t;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"((uint16_t)v) : "memory");
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_decode_fp8_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap panel_map) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  grid_launch_dependents();  // the combine may be launched behind this grid right away
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int32_t* slots_ring = reinterpret_cast<int32_t*>(smem + kOffSlots);
  uint8_t* valid = smem + kOffValid;
  float* pre_ring = reinterpret_cast<float*>(smem + kOffPre);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t xbeg = tile_begin(blockIdx.x, p.total, p.G);
  const int64_t xend = tile_begin(blockIdx.x + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);

  if (tid == 0) {
    for (int i = 0; i < kOpBufs; ++i) {
      // per loader: one arrival with its TMA bytes, and one per row when the row's scale copy lands
      mbar_init(&bars[kBarOpFull + i], kLoaders + kRows);
      mbar_init(&bars[kBarOpEmpty + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarSFree + i], kSoftWarps);
    }
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(&bars[kBarPFull + i], kSoftWarps);
      mbar_init(&bars[kBarPvDone + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kBarIdxFull + i], 32);
      mbar_init(&bars[kBarIdxEmpty + i], kLoaders);
    }
    mbar_init(&bars[kBarQFull], kQWarps);
    mbar_init(&bars[kBarQEmpty], 1);
    mbar_init(&bars[kBarOFree], kSoftWarps);
    mbar_init(&bars[kBarDrain], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent (of the cache store, typically): the
  // index translation and the Q split read only this call's inputs and write
  // only shared memory, so they start at once; every other role reads the
  // cache or writes global memory, and first waits for the preceding grid.
  if (warp != kIndexWarp && (warp < kQWarp0 || warp >= kQWarp0 + kQWarps)) grid_dependency_wait();

#define SMLA_WAIT(bar_idx, parity) mbar_wait(&bars[(bar_idx)], (parity), abort_flag, p.status, kDevWaitTimeout)

  if (warp == kIndexWarp) {
    // ------------------------------------------------------------ index translation
    // The next tile's indices are loaded before this tile's block-table reads,
    // so each tile costs about one memory round trip.
    int32_t cur[2], nxt[2], req_cur = 0, req_nxt = 0;
    auto load_idx = [&](int tl, int32_t (&v)[2], int32_t& rq) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      rq = __ldg(p.req_id + ti.t);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = ti.kt * kRows + lane + 32 * i;
        v[i] = k < p.K ? __ldg(p.indices + (int64_t)ti.t * p.K + k) : -1;
      }
    };
    if (n_local > 0) load_idx(0, cur, req_cur);
    for (int tl = 0; tl < n_local; ++tl) {
      if (tl + 1 < n_local) load_idx(tl + 1, nxt, req_nxt);
      const int b4 = tl & 3;
      if (tl >= 4 && !SMLA_WAIT(kBarIdxEmpty + b4, ((tl >> 2) + 1) & 1)) break;
#pragma unroll
      for (int i = 0; i < 2; ++i)
        slots_ring[b4 * kRows + lane + 32 * i] = translate_slot(cur[i], req_cur, p.block_table, p.R, p.MB, p.NB);
      mbar_arrive(&bars[kBarIdxFull + b4]);
      if (lane == 0) SMLA_TRACE_SET(tl, kEvIdx);
#pragma unroll
      for (int i = 0; i < 2; ++i) cur[i] = nxt[i];
      req_cur = req_nxt;
    }
  } else if (warp >= kLoadWarp0 && warp < kLoadWarp0 + kLoaders) {
    // ------------------------------------------------------------ loaders
    // Loader lw gathers rows 16 lw .. 16 lw + 15 of every tile: 4 groups of 4
    // rows x 5 TMA copies (code panels 0..3, RoPE panel), lane 5 g + b
    // issuing copy b of group g, and each row's 16 bytes of scales as one
    // cp.async by lane r (zero-filled for an invalid row), which keeps these
    // small copies out of the SM's TMA queue.  Its arrival on the tile's full
    // barrier carries the TMA bytes of its 16 rows and follows its writes of
    // the rows' valid flags; each scale copy arrives there when it lands.
    const int lw = warp - kLoadWarp0;
    const int grp = lane / 5, box = lane % 5;  // lanes 0..19 issue TMA copies
    const int r_g = 16 * lw + 4 * grp;         // tile row of the lane's group
    int last_ob = -1, last_use = 0;
    for (int tl = 0; tl < n_local; ++tl) {
      const int b4 = tl & 3, ob = tl % kOpBufs, use = tl / kOpBufs;
      if (!SMLA_WAIT(kBarIdxFull + b4, (tl >> 2) & 1)) break;
      const int32_t slot = lane < 16 ? slots_ring[b4 * kRows + 16 * lw + lane] : -1;
      const uint32_t vmask = __ballot_sync(kFullMask, slot >= 0);
      const int row = slot >= 0 ? slot : -1;
      const int g0 = __shfl_sync(kFullMask, row, (4 * grp) & 31), g1 = __shfl_sync(kFullMask, row, (4 * grp + 1) & 31);
      const int g2 = __shfl_sync(kFullMask, row, (4 * grp + 2) & 31), g3 = __shfl_sync(kFullMask, row, (4 * grp + 3) & 31);
      if (lane == 0) mbar_arrive(&bars[kBarIdxEmpty + b4]);  // this quarter's slots read
      if (use >= 1 && !SMLA_WAIT(kBarOpEmpty + ob, (use + 1) & 1)) break;
      if (lane == 0 && lw == 0) SMLA_TRACE_SET(tl, kEvOpEmpty);
      if (lane < 16) valid[ob * kRows + 16 * lw + lane] = (uint8_t)((vmask >> lane) & 1u);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBarOpFull + ob], 16 * (4 * 128 + 128));
      __syncwarp();
      const uint32_t op = smem_u32(smem + kOffOp + ob * kOpBuf);
      if (lane < 20) {
        const uint32_t in_panel = (uint32_t)((r_g >> 3) * 1024 + (r_g & 7) * 128);
        const uint32_t dst = box < 4 ? op + box * kPanel + in_panel : op + kOpRope + in_panel;
        tma_gather4(dst, &panel_map, box < 4 ? 128 * box : kRopeOff, g0, g1, g2, g3, &bars[kBarOpFull + ob]);
      }
      if (lane < 16) {
        const int r = 16 * lw + lane;
        const uint8_t* src = slot >= 0 ? p.cache + (int64_t)slot * kRowBytes + kScaleOff : p.cache;
        cp_async_16_zfill(op + kOpScale + (uint32_t)((r >> 2) * 128 + (r & 3) * 16), src, slot >= 0 ? 16u : 0u);
        cp_async_mbar_arrive_noinc(&bars[kBarOpFull + ob]);
      }
      if (lane == 0 && lw == 0) SMLA_TRACE_SET(tl, kEvIssue);
      last_ob = ob;
      last_use = use;
    }
    // No copy may still be landing in shared memory when the CTA exits (only
    // possible after an abort; the consumers have waited for every tile otherwise).
    if (last_ob >= 0) mbar_wait_drain(&bars[kBarOpFull + last_ob], last_use & 1);
  } else if (warp >= kQWarp0 && warp < kQWarp0 + kQWarps) {
    // ------------------------------------------------------------ Q preparation
    // 4 threads per head: thread part owns NoPE columns [128 part, 128 part +
    // 128) (code panel `part`) and RoPE chunks 2 part, 2 part + 1.  Head h is
    // stored in operand row n = q_row_of_head(h) (hi) and 16 + n (lo).
    // q * 2^s_hg = hi + lo in e4m3 with s_hg chosen so that the largest
    // |q * 2^s_hg| over the thread's 128 columns (scale group g = part) is at
    // most 448.
    // One Q buffer: the next segment's q is loaded into registers while the
    // current one is in use, and converted once the buffer is released.
    const int qt = tid - 32 * kQWarp0;  // 0..63
    const int h = qt >> 2, part = qt & 3;
    const int qrow = q_row_of_head(h);
    uint4 v[16], rope0, rope1;
    auto load_q = [&](int tl) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)ti.t * p.H + ti.hg * HG + h) * kDqk);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __ldg(src + 16 * part + i);
      rope0 = __ldg(src + 64 + 2 * part);
      rope1 = __ldg(src + 64 + 2 * part + 1);
    };
    int tl = 0, seg = 0;
    if (n_local > 0) load_q(0);
    while (tl < n_local) {
      if (seg >= 1 && !SMLA_WAIT(kBarQEmpty, (seg - 1) & 1)) break;
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[k] << 16)), fabsf(__uint_as_float(w4[k] & 0xFFFF0000u))));
      }
      // one prescale per (head, scale group): the group's own largest |q| sets it
      int sh = 0;
      if (amax > 0.f) {
        int e;
        frexpf(448.f / amax, &e);  // 448 / amax = m * 2^e, m in [0.5, 1)
        sh = e - 1;
      }
      const float pre = ldexpf(1.f, sh);
      const uint32_t qpanel = smem_u32(smem + kOffQ + part * kQPanel);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {  // 16 codes per chunk = two uint4 of bf16
        uint32_t hi[4], lo[4];
        const uint32_t w8[8] = {v[2 * ch].x,     v[2 * ch].y,     v[2 * ch].z,     v[2 * ch].w,
                                v[2 * ch + 1].x, v[2 * ch + 1].y, v[2 * ch + 1].z, v[2 * ch + 1].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t h0, l0, h1, l1;
          split2(__uint_as_float(w8[2 * k] << 16) * pre, __uint_as_float(w8[2 * k] & 0xFFFF0000u) * pre, h0, l0);
          split2(__uint_as_float(w8[2 * k + 1] << 16) * pre, __uint_as_float(w8[2 * k + 1] & 0xFFFF0000u) * pre, h1, l1);
          hi[k] = h0 | (h1 << 16);
          lo[k] = l0 | (l1 << 16);
        }
        sts128(qpanel + sw128_chunk(32, qrow, ch), make_uint4(hi[0], hi[1], hi[2], hi[3]));
        sts128(qpanel + sw128_chunk(32, 16 + qrow, ch), make_uint4(lo[0], lo[1], lo[2], lo[3]));
      }
      const uint32_t qrope = smem_u32(smem + kOffQ + kQRope);
      sts128(qrope + sw128_chunk(HG, qrow, 2 * part), rope0);
      sts128(qrope + sw128_chunk(HG, qrow, 2 * part + 1), rope1);
      pre_ring[((seg & 3) * 4 + part) * HG + qrow] = ldexpf(1.f, -sh);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarQFull]);
      if (qt == 0) SMLA_TRACE_SET(tl, kEvQReady);
      // the next segment starts at the next tile with top-k tile index 0
      do {
        ++tl;
      } while (tl < n_local && tile_info(p, xbeg + tl, xbeg, xend).kt != 0);
      if (tl < n_local) load_q(tl);
      ++seg;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tensor-core issuer
    // Polls (never blocks on) the next P' for P.V, then the next operand tile
    // + Q + free S buffer for QK^T (an S buffer is free once the softmax has
    // read the tile two before out of it).  P.V goes first: its completion
    // frees the operand tile and the P buffer that the other roles wait for.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_qk8 = idesc_e4m3(64, 32, 0, 0);
      constexpr uint32_t id_qkr = make_idesc_bf16(64, HG, 0, 0);
      constexpr uint32_t id_pv = idesc_e4m3(128, 32, 1, 1);
      const uint32_t op0 = smem_u32(smem + kOffOp), q0 = smem_u32(smem + kOffQ), p0 = smem_u32(smem + kOffP);
      // Shared-memory descriptors are built once; an operand at a byte offset
      // o from a base is that descriptor + o / 16 (the start-address field holds
      // bits 4..17 of the address, and no offset here carries out of it).
      const uint64_t dK0 = make_sdesc(op0, 16, 1024, kLayoutSw128);
      const uint64_t dQ = make_sdesc(q0, 16, 1024, kLayoutSw128);
      const uint64_t dV0 = make_sdesc(op0, kPanel, 1024, kLayoutSw128);
      const uint64_t dP0 = make_sdesc(p0, 256, 128, kLayoutNone);
      int seg_q = 0, seg_o = 0, next_qk = 0, next_pv = 0;
      // top-k tile index within its unit of the next QK^T / P.V tile (advanced
      // incrementally: no divisions in the polling loop)
      const int kt0 = (int)(xbeg % p.nt);
      int kt_qk = kt0, kt_pv = kt0, ob_qk = 0, ob_pv = 0, pb_pv = 0, pb_use = 0;
      uint64_t t_idle = 0;
      uint32_t idle_polls = 0;
      while (next_pv < n_local) {
        bool progressed = false;
        if (next_pv < next_qk) {
          const int tl = next_pv;
          const bool seg_start = tl == 0 || kt_pv == 0;
          const int pb = pb_pv;
          const bool o_ok = !seg_start || seg_o == 0 || mbar_test_wait(&bars[kBarOFree], (seg_o - 1) & 1);
          if (o_ok && mbar_test_wait(&bars[kBarPFull + pb], pb_use & 1)) {
            SMLA_TRACE_SET(tl, kEvPvSeen);
            if (seg_start) ++seg_o;
            tc_fence_after();
            const uint64_t dv = dV0 + (uint64_t)((ob_pv * kOpBuf) >> 4), dp = dP0 + (uint64_t)((pb * kPBuf) >> 4);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
              for (int k = 0; k < 2; ++k)
                // A = codes^T (value column c x row j), MN-major; B = P'_q (row j x 32), MN-major
                mma_f8(tmem + kOCol + 32 * q, dv + ((q * kPanel + 4096 * k) >> 4), dp + ((q * kPGroup + 1024 * k) >> 4),
                       id_pv, (seg_start && k == 0) ? 0u : 1u);
            }
            mma_commit(&bars[kBarOpEmpty + ob_pv]);
            mma_commit(&bars[kBarPvDone + pb]);
            SMLA_TRACE_SET(tl, kEvPv);
            ++next_pv;
            kt_pv = kt_pv + 1 == p.nt ? 0 : kt_pv + 1;
            ob_pv = ob_pv + 1 == kOpBufs ? 0 : ob_pv + 1;
            if (++pb_pv == kPBufs) {
              pb_pv = 0;
              ++pb_use;
            }
            progressed = true;
          }
        }
        if (next_qk < n_local &&
            (next_qk < 2 || mbar_test_wait(&bars[kBarSFree + (next_qk & 1)], ((next_qk - 2) >> 1) & 1))) {
          const int tl = next_qk;
          const bool seg_start = tl == 0 || kt_qk == 0;
          const bool seg_end = tl == n_local - 1 || kt_qk == p.nt - 1;
          const int sbuf = tl & 1;
          const int seg = seg_start ? seg_q : seg_q - 1;
          const bool q_ok = !seg_start || mbar_test_wait(&bars[kBarQFull], seg & 1);
          if (q_ok && mbar_test_wait(&bars[kBarOpFull + ob_qk], (tl / kOpBufs) & 1)) {
            SMLA_TRACE_SET(tl, kEvQkSeen);
            if (seg_start) ++seg_q;
            tc_fence_after();
            const uint64_t dk = dK0 + (uint64_t)((ob_qk * kOpBuf) >> 4);
            const uint32_t sb = tmem + sbuf * kSCols;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f8(sb + 32 * g, dk + ((g * kPanel + 32 * k) >> 4), dQ + ((g * kQPanel + 32 * k) >> 4), id_qk8,
                       k > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(sb + 128, dk + ((kOpRope + 32 * k) >> 4), dQ + ((kQRope + 32 * k) >> 4), id_qkr, k > 0 ? 1u : 0u);
            mma_commit(&bars[kBarSFull + sbuf]);
            if (seg_end) mma_commit(&bars[kBarQEmpty]);
            SMLA_TRACE_SET(tl, kEvQk);
            ++next_qk;
            kt_qk = kt_qk + 1 == p.nt ? 0 : kt_qk + 1;
            ob_qk = ob_qk + 1 == kOpBufs ? 0 : ob_qk + 1;
            progressed = true;
          }
        }
        if (progressed) {
          t_idle = 0;
          idle_polls = 0;
        } else if ((++idle_polls & 255u) == 0u) {
          // the abort flag and the clock are looked at every 256 idle polls only:
          // reading %globaltimer on every poll slows the reaction to ready work
          if (*abort_flag) break;
          const uint64_t now = globaltimer_ns();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > kWaitLimitNs) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, kDevWaitTimeout);
            break;
          }
        }
      }
      // every issued tensor-core operation completes before tensor memory is released
      if (next_qk > 0) {
        mma_commit(&bars[kBarDrain]);
        mbar_wait_drain(&bars[kBarDrain], 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue (warps 0..7)
    // QK^T with M = 64 leaves tile row r in TMEM lane 32 (r / 16) + r % 16.
    // Warp w reads lane quarter qd = w % 4 and the head columns of half
    // hh = w / 4 with the 16x256b shape: thread (w, lane) holds rows
    // r0 = 16 qd + lane / 4 and r1 = r0 + 8 of columns nA = 8 hh + 2 (lane % 4)
    // and nA + 1; item k (0..3) is row k >> 1 of column nA + (k & 1).  Each
    // thread keeps the running state of its 2 columns.  The two halves share
    // nothing but the barriers on S, P' and O: each decides its own rescales
    // and rescales its own columns of O.  For the P.V output (M = 128) thread
    // lane of warp w owns value column 32 qd + lane of each chunk, for the
    // columns of its half.
    const int w = warp, qd = w & 3, hh = w >> 2;
    const int c4 = lane & 3;
    const int r0 = 16 * qd + (lane >> 2), r1 = r0 + 8;
    const int nA = 8 * hh + 2 * c4;
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    const uint32_t p0 = smem_u32(smem + kOffP);
    const int bar_id = 1 + hh;  // named barrier of the half (4 warps)
    float* red_max = reinterpret_cast<float*>(smem + kOffRedMax);
    float* red_sc = reinterpret_cast<float*>(smem + kOffRedSc);
    float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
    float m2[2], l2[2], ip2[4][2], Rq[4];
    SMLA_CLK_DECL;
    int seg = -1, seg_first_kt = 0, n_seg_tiles = 0;
    bool dead = false;
    // waits of this role keep `dead` warp-uniform: the tensor-memory accesses
    // and shuffles it guards are warp-collective
    auto wait_s = [&](int bar_idx, uint32_t parity) {
      if (!dead) dead = !SMLA_WAIT(bar_idx, parity);
      dead = __any_sync(kFullMask, dead);
    };
    TileInfo ti = tile_info(p, xbeg, xbeg, xend);
    for (int tl = 0; tl < n_local; ++tl) {
      if (tl > 0) {  // advance the tile position without divisions
        ti.seg_start = ++ti.kt == p.nt;
        if (ti.seg_start) {
          ti.kt = 0;
          ++ti.u;
          if (++ti.hg == p.n_hg) {
            ti.hg = 0;
            ++ti.t;
          }
        }
        ti.seg_end = tl == n_local - 1 || ti.kt == p.nt - 1;
      }
      const int ob = tl % kOpBufs, sbuf = tl & 1, pb = tl % kPBufs, puse = tl / kPBufs;
      if (ti.seg_start) {
        ++seg;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          m2[e] = -INFINITY;
          l2[e] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) Rq[g] = 0.f;
        seg_first_kt = ti.kt;
        n_seg_tiles = 0;
      }
      SMLA_CLK_MARK(11);
      wait_s(kBarOpFull + ob, (tl / kOpBufs) & 1);  // row flags and scales
      if (tid == 0) SMLA_TRACE_SET(tl, kEvOpFull);
      SMLA_CLK_MARK(12);
      wait_s(kBarSFull + sbuf, (tl >> 1) & 1);
      if (tid == 0) SMLA_TRACE_SET(tl, kEvSoftStart);
      SMLA_CLK_START();
      tc_fence_after();
      if (ti.seg_start) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float2 v = *reinterpret_cast<const float2*>(pre_ring + ((seg & 3) * 4 + g) * HG + nA);
          ip2[g][0] = v.x;
          ip2[g][1] = v.y;
        }
      }
      const bool ok0 = !dead && valid[ob * kRows + r0] != 0;
      const bool ok1 = !dead && valid[ob * kRows + r1] != 0;
      const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
      const uint8_t* scl = smem + kOffOp + ob * kOpBuf + kOpScale;
      const float4 s0 = ok0 ? *reinterpret_cast<const float4*>(scl + (r0 >> 2) * 128 + (r0 & 3) * 16) : zero4;
      const float4 s1 = ok1 ? *reinterpret_cast<const float4*>(scl + (r1 >> 2) * 128 + (r1 & 3) * 16) : zero4;
      const float sc0[4] = {s0.x, s0.y, s0.z, s0.w};
      const float sc1[4] = {s1.x, s1.y, s1.z, s1.w};
      // logits (log2 units): sum_g scale_g 2^-s_hg (S_g,hi + S_g,lo) + S_rope
      float sl[4];
      {
        const uint32_t sa = tmem + lane_base + sbuf * kSCols + 8 * hh;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (!dead) {
          uint32_t hi[4][4], lo[4][4], rp[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            tmem_ld_16x256b_x1(sa + 32 * g, hi[g]);
            tmem_ld_16x256b_x1(sa + 32 * g + 16, lo[g]);
          }
          tmem_ld_16x256b_x1(sa + 128, rp);
          tmem_ld_wait();
          // S of this tile is in registers: its buffer may take QK^T of tile tl + 2
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarSFree + sbuf]);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            reg_fence4(hi[g]);
            reg_fence4(lo[g]);
          }
          reg_fence4(rp);
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              acc[k] = fmaf(((k >> 1) ? sc1[g] : sc0[g]) * ip2[g][k & 1],
                            __uint_as_float(hi[g][k]) + __uint_as_float(lo[g][k]), acc[k]);
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[k] += __uint_as_float(rp[k]);
        } else if (lane == 0) {
          mbar_arrive(&bars[kBarSFree + sbuf]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) sl[k] = ((k >> 1) ? ok1 : ok0) ? acc[k] * p.scale_log2 : -INFINITY;
      }
      if (tid == 0) SMLA_TRACE_SET(tl, kEvSoftLogits);
      SMLA_CLK_MARK(0);
      // tile maxima: per column (logits) and per scale group (scales), across the 64 rows
      float* redm = red_max + (tl & 1) * 4 * HG;
      float* reds = red_sc + ((tl & 1) * 2 + hh) * 4 * 4;
      {
        float t2[2] = {fmaxf(sl[0], sl[2]), fmaxf(sl[1], sl[3])};
        float s4[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) s4[g] = fmaxf(sc0[g], sc1[g]);
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
#pragma unroll
          for (int e = 0; e < 2; ++e) t2[e] = fmaxf(t2[e], __shfl_xor_sync(kFullMask, t2[e], off));
#pragma unroll
          for (int g = 0; g < 4; ++g) s4[g] = fmaxf(s4[g], __shfl_xor_sync(kFullMask, s4[g], off));
        }
        if (lane < 4) *reinterpret_cast<float2*>(redm + qd * HG + nA) = make_float2(t2[0], t2[1]);
        if (lane == 0) *reinterpret_cast<float4*>(reds + qd * 4) = make_float4(s4[0], s4[1], s4[2], s4[3]);
      }
      named_bar_sync(bar_id, 128);
      if (tid == 0) SMLA_TRACE_SET(tl, kEvSoftBar);
      SMLA_CLK_MARK(1);
      // running maxima of the own columns (lazy: refreshed only when the tile
      // maximum exceeds them by more than kMaxSlack) and power-of-two bounds
      // of the scale groups
      float alpha2[2], beta[4];
      bool up_any = false, rq_changed = false;
      {
        float2 a[4];
        float4 c[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          a[v] = *reinterpret_cast<const float2*>(redm + v * HG + nA);
          c[v] = *reinterpret_cast<const float4*>(reds + 4 * v);
        }
        const float tmax[2] = {fmaxf(fmaxf(a[0].x, a[1].x), fmaxf(a[2].x, a[3].x)),
                               fmaxf(fmaxf(a[0].y, a[1].y), fmaxf(a[2].y, a[3].y))};
        const float smax[4] = {fmaxf(fmaxf(c[0].x, c[1].x), fmaxf(c[2].x, c[3].x)), fmaxf(fmaxf(c[0].y, c[1].y), fmaxf(c[2].y, c[3].y)),
                               fmaxf(fmaxf(c[0].z, c[1].z), fmaxf(c[2].z, c[3].z)), fmaxf(fmaxf(c[0].w, c[1].w), fmaxf(c[2].w, c[3].w))};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float nm = fmaxf(m2[e], tmax[e]);
          const bool up = nm > m2[e] + kMaxSlack;
          const float mnew = nm + kMaxOvershoot;
          alpha2[e] = up ? ex2_approx(m2[e] - mnew) : 1.f;
          m2[e] = up ? mnew : m2[e];
          l2[e] *= alpha2[e];
          up_any |= up;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const bool grow = smax[g] > Rq[g];
          const float rn = grow ? pow2_ceil(smax[g]) : Rq[g];
          beta[g] = (grow && Rq[g] > 0.f) ? Rq[g] * rcp_pow2(rn) : 1.f;
          rq_changed |= grow && Rq[g] > 0.f;
          Rq[g] = rn;
        }
      }
      // every warp of a half sees all 8 of its columns (lanes 0..3) and the same
      // shared maxima: the decision is uniform over the half
      const bool rescale = __any_sync(kFullMask, up_any) || rq_changed;
#ifdef SMLA_TRACE
      if (n_seg_tiles > 0) {
        clk_acc[8] += __any_sync(kFullMask, up_any) ? 1u : 0u;
        clk_acc[9] += rq_changed ? 1u : 0u;
        clk_acc[10] += 1u;
      }
#endif
      SMLA_CLK_MARK(2);
      if (rescale && n_seg_tiles > 0) {
        // O^T holds this segment's earlier P.V: wait for the latest and rescale
        // this half's columns in place (column 8 hh + j: alpha of lane j / 2)
        float alpha[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) alpha[j] = __shfl_sync(kFullMask, alpha2[j & 1], j >> 1);
        wait_s(kBarPvDone + (tl - 1) % kPBufs, ((tl - 1) / kPBufs) & 1);  // P.V(tl - 1) and all before
        if (!dead) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t oh[8], ol[8];
            const uint32_t addr = tmem + lane_base + kOCol + 32 * q + 8 * hh;
            tmem_ld8(addr, oh);
            tmem_ld8(addr + 16, ol);
            tmem_ld_wait();
            reg_fence8(oh);
            reg_fence8(ol);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float f = alpha[j] * beta[q];
              oh[j] = __float_as_uint(__uint_as_float(oh[j]) * f);
              ol[j] = __float_as_uint(__uint_as_float(ol[j]) * f);
            }
            tmem_st8(addr, oh);
            tmem_st8(addr + 16, ol);
          }
          tmem_st_wait();
        }
      }
      SMLA_CLK_MARK(3);
      // probabilities and running sums
      float pr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pr[k] = ((k >> 1) ? ok1 : ok0) ? ex2_approx(sl[k] - m2[k & 1]) : 0.f;
        l2[k & 1] += pr[k];
      }
      SMLA_CLK_MARK(4);
      if (tl >= kPBufs) wait_s(kBarPvDone + pb, (puse + 1) & 1);  // P buffer free: P.V(tl - 3) done
      if (tid == 0) SMLA_TRACE_SET(tl, kEvSoftPWait);
      SMLA_CLK_MARK(5);
      // P'_q = kPScale * p * scale_q / R_q as e4m3 hi + lo: MN-major core
      // matrices of 8 rows x 16 codes (columns), hi and lo blocks 128 B apart,
      // row blocks 256 B apart
      if (!dead) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float inv_r = Rq[g] > 0.f ? kPScale * rcp_pow2(Rq[g]) : 0.f;
#pragma unroll
          for (int rho = 0; rho < 2; ++rho) {
            const int r = rho ? r1 : r0;
            const float f = (rho ? sc1[g] : sc0[g]) * inv_r;
            uint32_t hw, lw;
            split2_f16(pr[2 * rho] * f, pr[2 * rho + 1] * f, hw, lw);
            const uint32_t base = p0 + pb * kPBuf + g * kPGroup + (r >> 3) * 256 + (r & 7) * 16 + nA;
            sts16(base, hw);
            sts16(base + 128, lw);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !dead) mbar_arrive(&bars[kBarPFull + pb]);
      if (tid == 0) SMLA_TRACE_SET(tl, kEvSoftDone);
      SMLA_CLK_MARK(6);
      ++n_seg_tiles;

      if (ti.seg_end) {
        {
          float v2[2] = {l2[0], l2[1]};
#pragma unroll
          for (int off = 4; off <= 16; off <<= 1)
#pragma unroll
            for (int e = 0; e < 2; ++e) v2[e] += __shfl_xor_sync(kFullMask, v2[e], off);
          if (lane < 4) *reinterpret_cast<float2*>(red_sum + qd * HG + nA) = make_float2(v2[0], v2[1]);
        }
        named_bar_sync(bar_id, 128);
        wait_s(kBarPvDone + pb, puse & 1);  // last P.V of the segment
        tc_fence_after();
        const bool full = (seg_first_kt == 0) && (ti.kt == p.nt - 1);
        const int64_t slot = (int64_t)blockIdx.x + ti.u;
        const int64_t row0 = (int64_t)ti.t * p.H + ti.hg * HG;
        float inv[8];
#pragma unroll
        for (int j4 = 0; j4 < 2; ++j4) {
          const int n0 = 8 * hh + 4 * j4;
          const float4 a0 = *reinterpret_cast<const float4*>(red_sum + n0);
          const float4 a1 = *reinterpret_cast<const float4*>(red_sum + HG + n0);
          const float4 a2 = *reinterpret_cast<const float4*>(red_sum + 2 * HG + n0);
          const float4 a3 = *reinterpret_cast<const float4*>(red_sum + 3 * HG + n0);
          const float lt[4] = {(a0.x + a1.x) + (a2.x + a3.x), (a0.y + a1.y) + (a2.y + a3.y),
                               (a0.z + a1.z) + (a2.z + a3.z), (a0.w + a1.w) + (a2.w + a3.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            inv[4 * j4 + e] = lt[e] > 0.f ? __frcp_rn(lt[e]) : 0.f;
            // lse of column n0 + e from the thread that holds its running maximum
            const int n = n0 + e;
            if (qd == 0 && lane == ((n & 7) >> 1)) {
              const float lse_v = lt[e] > 0.f ? (m2[n & 1] + log2f(lt[e])) * 0.69314718055994530942f : -INFINITY;
              const int h = head_of_col(n);
              if (full)
                p.lse[row0 + h] = lse_v;
              else
                p.part_lse[slot * HG + h] = lse_v;
            }
          }
        }
        if (!dead) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t ohi[8], olo[8];
            tmem_ld8(tmem + lane_base + kOCol + 32 * q + 8 * hh, ohi);
            tmem_ld8(tmem + lane_base + kOCol + 32 * q + 16 + 8 * hh, olo);
            tmem_ld_wait();
            reg_fence8(ohi);
            reg_fence8(olo);
            const int c = 128 * q + 32 * qd + lane;
            const float rs = Rq[q] * kPScaleInv;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int h = head_of_col(8 * hh + j);
              const float val = (__uint_as_float(ohi[j]) + __uint_as_float(olo[j])) * rs * inv[j];
              if (full)
                p.out[(row0 + h) * kDv + c] = __float2bfloat16_rn(val);
              else
                p.part_o[(slot * HG + h) * kDv + c] = val;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !dead) mbar_arrive(&bars[kBarOFree]);
        SMLA_CLK_MARK(7);
      }
    }
    SMLA_CLK_STORE();
  }
#undef SMLA_WAIT

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Tensor map of the cache viewed as a 2-D byte array [NB * 64 rows, 656
// bytes]: 128-byte boxes with the 128-byte swizzle (code and RoPE panels).
// Rows outside [0, NB * 64) read as zeros.
cudaError_t make_cache_map(const uint8_t* cache, int64_t NB, CUtensorMap* panel_map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)(NB * kBlock)};
  const cuuint64_t gstride[1] = {(cuuint64_t)kRowBytes};
  const cuuint32_t box_panel[2] = {128, 1}, es[2] = {1, 1};
  const CUresult r = enc(panel_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(cache), gdim, gstride,
                         box_panel, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

#ifdef SMLA_TRACE
extern "C" int smla_trace_set_fp8(unsigned long long* buf) {
  return (int)cudaMemcpyToSymbol(g_smla_trace_fp8, &buf, sizeof(buf));
}
#endif

AttnPlan plan_decode_fp8(int T, int H, int K, int num_splits, int num_sms) {
  if (wide_supported(H)) return plan_decode_wide(T, K, num_splits, num_sms);
  AttnPlan pl;
  pl.HG = HG;
  pl.n_hg = H / HG;
  pl.nt = K > 0 ? (K + kRows - 1) / kRows : 1;
  pl.units = (int64_t)T * pl.n_hg;
  pl.total = pl.units * pl.nt;
  int64_t G = num_splits > 0 ? pl.units * (int64_t)num_splits : (int64_t)num_sms;
  if (G > pl.total) G = pl.total;
  if (G < 1) G = 1;
  pl.G = (int)G;
  pl.need_combine = !(pl.total % pl.G == 0 && (pl.total / pl.G) % pl.nt == 0);
  const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
  const size_t lse_bytes = (size_t)(((n_slots * HG * 4) + 255) / 256) * 256;
  pl.ws_bytes = kWsStatusBytes + lse_bytes + (size_t)n_slots * HG * kDv * 4;
  return pl;
}

cudaError_t launch_decode_fp8(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (plan.HG == 128) return launch_decode_wide(a, plan, stream);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int64_t n_slots = (int64_t)plan.G + plan.units - 1;
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.cache = a.cache;
  p.indices = a.indices;
  p.block_table = a.block_table;
  p.req_id = a.req_id;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = reinterpret_cast<int*>(ws);
  p.part_lse = reinterpret_cast<float*>(ws + kWsStatusBytes);
  p.part_o = reinterpret_cast<float*>(ws + kWsStatusBytes + ((n_slots * HG * 4 + 255) / 256) * 256);
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.T = a.T;
  p.H = a.H;
  p.K = a.K;
  p.R = a.R;
  p.MB = a.MB;
  p.NB = a.NB;
  p.n_hg = plan.n_hg;
  p.nt = plan.nt;
  p.total = plan.total;
  p.G = plan.G;
  CUtensorMap panel_map;
  cudaError_t em = make_cache_map(a.cache, a.NB, &panel_map);
  if (em != cudaSuccess) return em;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.G, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, sparse_mla_decode_fp8_kernel, p, panel_map);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  e = launch_combine<HG>(p.part_o, p.part_lse, p.out, p.lse, p.H, p.n_hg, p.nt, p.total, p.G, plan.units, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace smla
